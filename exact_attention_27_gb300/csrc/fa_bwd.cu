// Backward pass of exact attention on sm_103a ("L'attention fusionnee",
// section "La passe arriere : recalculer plutot que garder").
//
//   B1  D = rowsum(dO o O), one fp32 value per query row (a memory-bound
//       reduction run before everything else).
//   B2  per key tile: rebuild P from the saved L, then dV, dS, dK, dQ.
//   B3  dQ accumulator (fp32) -> bf16, times scale.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

// ------------------------------------------------------------------ B1
// D / 8 threads per row, each loading 16 bytes of O and 16 bytes of dO;
// the partial sums of a row are combined with warp shuffles.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const uint4* __restrict__ o,
                                                         const uint4* __restrict__ dO,
                                                         float* __restrict__ out, long long rows) {
  constexpr int TPR = D / 8;  // threads per row: 8 or 16, aligned within a warp
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = tid / TPR;
  const int part = static_cast<int>(tid % TPR);
  float acc = 0.0f;
  if (row < rows) {
    const uint4 a = __ldg(o + row * TPR + part);
    const uint4 g = __ldg(dO + row * TPR + part);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w};
    const uint32_t gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 af = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[t]));
      const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[t]));
      acc = fmaf(af.x, gf.x, acc);
      acc = fmaf(af.y, gf.y, acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) out[row] = acc;
}

// ------------------------------------------------------------------ B3
__global__ void __launch_bounds__(256) dq_finalize_kernel(const float4* __restrict__ acc,
                                                          uint4* __restrict__ dq, long long n8,
                                                          float scale) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = __ldg(acc + 2 * i);
  const float4 b = __ldg(acc + 2 * i + 1);
  dq[i] = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                     pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
}

}  // namespace

cudaError_t launch_preprocess(const void* o, const void* dO, float* Dout, long long rows, int d,
                              cudaStream_t stream) {
  const long long threads = rows * (d / 8);
  const long long blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (d == 64)
    preprocess_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint4*>(o), static_cast<const uint4*>(dO), Dout, rows);
  else
    preprocess_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint4*>(o), static_cast<const uint4*>(dO), Dout, rows);
  return cudaGetLastError();
}

cudaError_t launch_dq_finalize(const float* dq_acc, void* dq, long long n, float scale,
                               cudaStream_t stream) {
  const long long n8 = n / 8;  // n is a multiple of 64
  const long long blocks = (n8 + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  dq_finalize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(dq_acc), static_cast<uint4*>(dq), n8, scale);
  return cudaGetLastError();
}

cudaError_t launch_backward(const BwdMaps&, const float*, const float*, float*, void*, void*,
                            const AttnShape&, uint32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace fa
