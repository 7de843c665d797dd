// C ABI of the exact-attention library (declared in include/fa.h): argument
// validation, tensor-map encoding, dispatch to the kernels, error reporting.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace {

// Bits set by kernels whose bounded waits ran out (one word per device).
__device__ uint32_t g_fa_error_word;

// Caller-owned events recorded around the backward main kernel (timing hook).
cudaEvent_t g_bwd_before = nullptr;
cudaEvent_t g_bwd_after = nullptr;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Device address of g_fa_error_word on the current device.
uint32_t* error_word() { return static_cast<uint32_t*>(fa::symbol_address_cached(g_fa_error_word)); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [planes][rows][cols] tensor seen as 3-D (cols, rows, planes) with a box of
// box_cols x box_rows x 1.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr, int cols,
              int rows, long long planes, int box_cols, int box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * elem_bytes,
                           static_cast<cuuint64_t>(cols) * rows * elem_bytes};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_bf16(CUtensorMap* m, const void* ptr, int d, int N, long long planes) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, d, N, planes, 64, 128,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

// K or V of the forward: boxes of one key tile (64 rows when d = 256, else 128).
bool make_kv_map_bf16(CUtensorMap* m, const void* ptr, int d, int N, long long planes) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, d, N, planes, 64,
                  d == 256 ? 64 : 128, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Encodes the maps and launches the bf16 forward (one CTA per query tile or
// pair of tiles, or a pair of CTAs at d = 128, whose K map has 64-row boxes).
cudaError_t forward_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                         const fa::AttnShape& s, uint32_t* err, cudaStream_t stream) {
  const long long qplanes = static_cast<long long>(s.B) * s.Hq;
  const long long kvplanes = static_cast<long long>(s.B) * s.Hkv;
  const bool pair = fa::forward_uses_pair(s);
  CUtensorMap tq, tk, tv;
  const bool ok = make_map_bf16(&tq, q, s.d, s.N, qplanes) &&
                  (pair ? make_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, s.d, s.keys(),
                                   kvplanes, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)
                        : make_kv_map_bf16(&tk, k, s.d, s.keys(), kvplanes)) &&
                  make_kv_map_bf16(&tv, v, s.d, s.keys(), kvplanes);
  if (!ok) return cudaErrorInvalidValue;
  return pair ? fa::launch_forward_pair(tq, tk, tv, o, lse, s, err, stream)
              : fa::launch_forward(tq, tk, tv, o, lse, s, err, stream);
}

// A single thread waits on an mbarrier that nothing will ever complete, with
// the caller's time limit, then records the timeout like the real kernels do.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = fa::smem_u32(&bar);
  fa::mbar_init(b, 1);
  fa::fence_barrier_init();
  const uint64_t t0 = fa::globaltimer_ns();
  while (!fa::mbar_try_wait(b, 0)) {
    if (fa::globaltimer_ns() - t0 > limit_ns) {
      atomicOr(err, fa::kErrTimeoutOther);
      return;
    }
  }
}

}  // namespace

namespace fa {

uint32_t* device_error_word() { return error_word(); }

fa_status validate_backward(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dO, const void* dq, const void* dk,
                            const void* dv, int B, int H_q, int H_kv, int N, int d, float scale,
                            int causal) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARGUMENT;
  const fa_status st = validate(B, H_q, H_kv, N, d, scale, causal);
  if (st != FA_OK) return st;
  const void* p16[] = {q, k, v, o, dO, dq, dk, dv};
  for (const void* p : p16)
    if (!aligned16(p)) return FA_ERR_INVALID_ARGUMENT;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_INVALID_ARGUMENT;
  return FA_OK;
}

bool backward_uses_two_kernels(int d, bool deterministic) { return deterministic || d == 256; }

size_t backward_scratch_bytes(int B, int H_q, int N, int d, bool deterministic,
                              size_t* acc_off) {
  const size_t rows = static_cast<size_t>(B) * H_q * N;
  const size_t d_bytes = rows * sizeof(float);
  if (backward_uses_two_kernels(d, deterministic)) {
    *acc_off = 0;
    return d_bytes;
  }
  *acc_off = (d_bytes + 1023) & ~static_cast<size_t>(1023);  // accumulator 1 KiB aligned
  return *acc_off + rows * d * sizeof(float);
}

fa_status enqueue_backward(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dO, void* dq, void* dk, void* dv,
                           const AttnShape& s, float* Dbuf, float* acc, bool deterministic,
                           bool timed, cudaStream_t stream) {
  uint32_t* err = error_word();
  if (!err) return FA_ERR_CUDA;
  const int d = s.d, N = s.N;
  const long long rows = static_cast<long long>(s.B) * s.Hq * N;
  const long long qplanes = static_cast<long long>(s.B) * s.Hq;
  const long long kvplanes = static_cast<long long>(s.B) * s.Hkv;
  const bool two = backward_uses_two_kernels(d, deterministic);
  if (!two && !acc) return FA_ERR_INVALID_ARGUMENT;
  BwdMaps m{};
  bool ok = make_map_bf16(&m.q, q, d, N, qplanes) && make_kv_map_bf16(&m.k, k, d, N, kvplanes) &&
            make_kv_map_bf16(&m.v, v, d, N, kvplanes) && make_map_bf16(&m.dO, dO, d, N, qplanes);
  if (ok && !two)
    ok = encode_map_f32_acc(&m.dq_acc, acc, d, N, qplanes) &&
         encode_map_f32_acc32(&m.dq_acc32, acc, d, N, qplanes);
  if (!ok) return FA_ERR_CUDA;
  // Main dK/dV kernel between the caller's timing events, if any.
  timed = timed && g_bwd_before && g_bwd_after;
  cudaError_t e = launch_preprocess(o, dO, Dbuf, rows, d, stream, two ? nullptr : acc);
  if (e == cudaSuccess && timed) e = cudaEventRecord(g_bwd_before, stream);
  if (e == cudaSuccess)
    e = d == 256 ? launch_backward_d256_kv(m, lse, Dbuf, dk, dv, s, err, stream)
                 : launch_backward(m, lse, Dbuf, acc, dk, dv, s, err, stream, !two);
  if (e == cudaSuccess && timed) e = cudaEventRecord(g_bwd_after, stream);
  if (e == cudaSuccess)
    e = two ? launch_backward_dq(m, lse, Dbuf, dq, s, err, stream)
            : launch_dq_finalize(acc, dq, rows * d, s.scale, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status validate(int B, int H_q, int H_kv, int N, int d, float scale, int causal) {
  if (B < 1 || H_q < 1 || H_kv < 1 || N < 1) return FA_ERR_INVALID_ARGUMENT;
  if (H_q % H_kv != 0) return FA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_INVALID_ARGUMENT;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARGUMENT;
  if (d != 64 && d != 96 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  const double elems = static_cast<double>(B) * H_q * N * d;
  if (elems >= 1099511627776.0) return FA_ERR_INVALID_ARGUMENT;  // 2^40
  if ((N + 127) / 128 > 65535) return FA_ERR_INVALID_ARGUMENT;   // grid.y limit
  return FA_OK;
}

bool encode_map_bf16(CUtensorMap* m, const void* ptr, int d, int N, long long planes) {
  return make_map_bf16(m, ptr, d, N, planes);
}

bool encode_map_f32_acc(CUtensorMap* m, const void* ptr, int d, int N, long long planes) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, d, N, planes, 32, 128,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

bool encode_map_f32_acc32(CUtensorMap* m, const void* ptr, int d, int N, long long planes) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, d, N, planes, 32, 32,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace fa

extern "C" {

fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H_q, int H_kv, int N, int d, float scale, int causal,
                     cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARGUMENT;
  const fa_status st = fa::validate(B, H_q, H_kv, N, d, scale, causal);
  if (st != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_INVALID_ARGUMENT;
  uint32_t* err = error_word();
  if (!err) return FA_ERR_CUDA;
  fa::AttnShape s{B, H_q, H_kv, N, d, scale, causal};
  return forward_bf16(q, k, v, o, lse, s, err, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_forward_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H_q, int H_kv, int N_q, int N_kv, int d, float scale, int causal,
                        int q_offset, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARGUMENT;
  fa_status st = fa::validate(B, H_q, H_kv, N_q, d, scale, causal);
  if (st != FA_OK) return st;
  if (N_kv < 1 || q_offset < 0) return FA_ERR_INVALID_ARGUMENT;
  if (static_cast<double>(q_offset) + N_q + 128 >= 2147483647.0) return FA_ERR_INVALID_ARGUMENT;
  if (static_cast<double>(B) * H_kv * N_kv * d >= 1099511627776.0) return FA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_INVALID_ARGUMENT;
  uint32_t* err = error_word();
  if (!err) return FA_ERR_CUDA;
  fa::AttnShape s{B, H_q, H_kv, N_q, d, scale, causal};
  s.Nk = N_kv;
  s.q_offset = q_offset;
  return forward_bf16(q, k, v, o, lse, s, err, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_forward_fp8(const void* q, const void* k, const void* v_t, void* o, float* lse,
                         int B, int H_q, int H_kv, int N, int d, float scale, float q_descale,
                         float k_descale, float v_descale, int causal, cudaStream_t stream) {
  if (!q || !k || !v_t || !o || !lse) return FA_ERR_INVALID_ARGUMENT;
  const fa_status st = fa::validate(B, H_q, H_kv, N, d, scale, causal);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  for (float f : {q_descale, k_descale, v_descale})
    if (!std::isfinite(f) || !(f > 0.0f)) return FA_ERR_INVALID_ARGUMENT;
  const float s_eff = scale * q_descale * k_descale;
  if (!std::isfinite(s_eff) || !(s_eff > 0.0f)) return FA_ERR_INVALID_ARGUMENT;
  if (N % 16 != 0) return FA_ERR_INVALID_ARGUMENT;  // V^T rows of N bytes: 16-byte strides
  if (!aligned16(q) || !aligned16(k) || !aligned16(v_t) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_INVALID_ARGUMENT;
  CUtensorMap tq, tk, tvt;
  if (!make_map(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q, d, N, static_cast<long long>(B) * H_q,
                128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, k, d, N, static_cast<long long>(B) * H_kv,
                128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&tvt, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, v_t, N, d,
                static_cast<long long>(B) * H_kv, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return FA_ERR_CUDA;
  uint32_t* err = error_word();
  if (!err) return FA_ERR_CUDA;
  fa::AttnShape s{B, H_q, H_kv, N, d, s_eff, causal};
  return fa::launch_forward_fp8(tq, tk, tvt, o, lse, s, v_descale, err, stream) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

fa_status fa_backward_preprocess(const void* o, const void* dO, float* D, long long rows, int d,
                                 cudaStream_t stream) {
  if (!o || !dO || !D || rows < 1) return FA_ERR_INVALID_ARGUMENT;
  if (d != 64 && d != 96 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (!aligned16(o) || !aligned16(dO) || (reinterpret_cast<uintptr_t>(D) & 3u))
    return FA_ERR_INVALID_ARGUMENT;
  return fa::launch_preprocess(o, dO, D, rows, d, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_backward(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                      int H_q, int H_kv, int N, int d, float scale, int causal,
                      cudaStream_t stream) {
  const fa_status st = fa::validate_backward(q, k, v, o, lse, dO, dq, dk, dv, B, H_q, H_kv, N, d,
                                             scale, causal);
  if (st != FA_OK) return st;
  size_t acc_off = 0;
  const size_t bytes = fa::backward_scratch_bytes(B, H_q, N, d, false, &acc_off);
  void* scratch = nullptr;
  if (cudaMallocAsync(&scratch, bytes, stream) != cudaSuccess) return FA_ERR_CUDA;
  float* Dbuf = static_cast<float*>(scratch);
  float* acc = acc_off ? reinterpret_cast<float*>(static_cast<char*>(scratch) + acc_off) : nullptr;
  fa::AttnShape s{B, H_q, H_kv, N, d, scale, causal};
  const fa_status r = fa::enqueue_backward(q, k, v, o, lse, dO, dq, dk, dv, s, Dbuf, acc,
                                           /*deterministic=*/false, /*timed=*/true, stream);
  const cudaError_t ef = cudaFreeAsync(scratch, stream);
  return r != FA_OK ? r : (ef == cudaSuccess ? FA_OK : FA_ERR_CUDA);
}

fa_status fa_backward_deterministic(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dO, void* dq, void* dk,
                                    void* dv, int B, int H_q, int H_kv, int N, int d, float scale,
                                    int causal, cudaStream_t stream) {
  const fa_status st = fa::validate_backward(q, k, v, o, lse, dO, dq, dk, dv, B, H_q, H_kv, N, d,
                                             scale, causal);
  if (st != FA_OK) return st;
  size_t acc_off = 0;
  const size_t bytes = fa::backward_scratch_bytes(B, H_q, N, d, true, &acc_off);
  void* scratch = nullptr;
  if (cudaMallocAsync(&scratch, bytes, stream) != cudaSuccess) return FA_ERR_CUDA;
  fa::AttnShape s{B, H_q, H_kv, N, d, scale, causal};
  const fa_status r = fa::enqueue_backward(q, k, v, o, lse, dO, dq, dk, dv, s,
                                           static_cast<float*>(scratch), nullptr,
                                           /*deterministic=*/true, /*timed=*/false, stream);
  const cudaError_t ef = cudaFreeAsync(scratch, stream);
  return r != FA_OK ? r : (ef == cudaSuccess ? FA_OK : FA_ERR_CUDA);
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension";
    case FA_ERR_CUDA: return "CUDA runtime error";
    case FA_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel ran out";
  }
  return "unknown status";
}

fa_status fa_last_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  uint32_t* err = error_word();
  if (!err) return FA_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, err, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return FA_ERR_CUDA;
  if (word == 0) return FA_OK;
  if (cudaMemsetAsync(err, 0, sizeof(word), stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_ERR_DEVICE_TIMEOUT;
}

fa_status fa_set_forward_tile_rows(int rows) {
  if (rows != 0 && rows != 128 && rows != 256 && rows != 512) return FA_ERR_INVALID_ARGUMENT;
  fa::set_forward_rows_per_cta(rows);
  return FA_OK;
}

int fa_forward_tile_rows_for(int B, int H_q, int H_kv, int N_q, int N_kv, int d, int causal,
                             int q_offset, int sms) {
  if (fa::validate(B, H_q, H_kv, N_q, d, 1.0f, causal) != FA_OK) return 0;
  if (N_kv < 1 || q_offset < 0 || sms < 1) return 0;
  fa::AttnShape s{B, H_q, H_kv, N_q, d, 1.0f, causal};
  s.Nk = N_kv;
  s.q_offset = q_offset;
  return fa::forward_rows_for(s, sms);
}

void fa_set_backward_events(cudaEvent_t before, cudaEvent_t after) {
  g_bwd_before = before;
  g_bwd_after = after;
}

fa_status fa_selftest_wait_timeout(int limit_ms, cudaStream_t stream) {
  if (limit_ms < 1 || limit_ms > 2000) return FA_ERR_INVALID_ARGUMENT;
  uint32_t* err = error_word();
  if (!err) return FA_ERR_CUDA;
  wait_timeout_selftest_kernel<<<1, 1, 0, stream>>>(static_cast<uint64_t>(limit_ms) * 1000000ull,
                                                    err);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
