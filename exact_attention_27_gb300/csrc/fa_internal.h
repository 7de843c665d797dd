// Internal interface between the C-ABI layer (fa_api.cu) and the kernel
// translation units.  Not installed; the public interface is include/fa.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>

#include "fa.h"

namespace fa {

struct AttnShape {
  int B, Hq, Hkv, N, d;  // N: query rows (and key rows unless Nk says otherwise)
  float scale;
  int causal;
  int Nk = 0;        // key/value rows; 0 means N
  int q_offset = 0;  // absolute position of query row 0 under the causal mask
  int keys() const { return Nk > 0 ? Nk : N; }
};

// Forward: q/k/v tensor maps (3-D: d, N, B*H; box 64 x 128 x 1; 128-byte
// swizzle; for d = 256 the k and v boxes are 64 x 64 x 1), outputs o (bf16)
// and lse (fp32).  Returns the launch status.
cudaError_t launch_forward(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           void* o, float* lse, const AttnShape& s, uint32_t* err,
                           cudaStream_t stream);
// FP8 forward, d = 128: q, k maps over e4m3 [.., N, 128] with 128 x 128-byte
// boxes, tvt over V^T e4m3 [.., 128, N_kv] with 128 x 128-byte boxes; s.scale
// already includes the Q and K descales, O is multiplied by v_descale.
cudaError_t launch_forward_fp8(const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tvt, void* o, float* lse, const AttnShape& s,
                               float v_descale, uint32_t* err, cudaStream_t stream);
// The forward with one query tile per CTA (fa_fwd_tile1.cu), d in {64, 128,
// 256}; launch_forward chooses it (always for d = 256).
cudaError_t launch_forward_tile1(const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, void* o, float* lse, const AttnShape& s,
                                 uint32_t* err, cudaStream_t stream);
// Launches kern<<<grid, block, smem, stream>>>(args...) as a programmatic
// dependent of the previous grid in the stream (the kernel must call
// grid_dependency_wait before reading what that grid writes).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Raises kernel Kern's dynamic shared-memory limit to `bytes` once per
// device instead of at every launch (the attribute call costs microseconds
// of host time; the setting belongs to the device's context, so each device
// ordinal below 64 is remembered separately and higher ordinals set it each
// time).
template <auto Kern>
cudaError_t set_smem_limit_once(int bytes) {
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launch-order grouping of query heads, shared by the forward kernels, the
// dQ kernel and the forward's tile-size estimate: whole GQA groups whose K/V
// (2 x keys x d elements of elem_bytes per K/V head) stay within about
// 48 MiB of the 129 MB L2; at least one group of G heads, at most n_heads.
inline long long heads_per_group(long long keys, int d, double elem_bytes, int G,
                                 long long n_heads) {
  const double kv_bytes = 2.0 * static_cast<double>(keys) * d * elem_bytes;
  long long kv_heads = static_cast<long long>(48.0 * 1024 * 1024 / kv_bytes);
  if (kv_heads < 1) kv_heads = 1;
  const long long hpg = kv_heads * G;
  return hpg < n_heads ? hpg : n_heads;
}

// Checks the sizes, scale and causal flag shared by every attention entry
// point: B, H_q, H_kv, N >= 1, H_q % H_kv == 0, scale finite and > 0, causal
// 0 or 1, B*H_q*N*d < 2^40 and at most 65535 query tiles per head
// (FA_ERR_INVALID_ARGUMENT); d in {64, 96, 128, 256} (else FA_ERR_UNSUPPORTED).
// Entry points that support fewer head dimensions check that afterwards.
fa_status validate(int B, int H_q, int H_kv, int N, int d, float scale, int causal);

// validate() plus the pointer checks of the backward entry points: every
// pointer non-null, 16-byte aligned (lse 4-byte aligned).
fa_status validate_backward(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dO, const void* dq, const void* dk,
                            const void* dv, int B, int H_q, int H_kv, int N, int d, float scale,
                            int causal);

// Whether the backward of head dimension d runs as two kernels (dK/dV, then
// dQ walking the key tiles in order; no dQ accumulator): always when
// `deterministic`, and at d = 256, whose only backward this is.
bool backward_uses_two_kernels(int d, bool deterministic);

// Scratch of one backward call: D (B*H_q*N fp32) and, for the single-kernel
// path, the fp32 dQ accumulator at byte offset *acc_off (1 KiB aligned);
// *acc_off = 0 when there is none.  Returns the total in bytes.
size_t backward_scratch_bytes(int B, int H_q, int N, int d, bool deterministic,
                              size_t* acc_off);

// Enqueues a validated backward pass on `stream`, given its scratch: Dbuf
// (B*H_q*N floats) and, unless the call runs as two kernels, acc (the fp32
// dQ accumulator, B*H_q*N*d floats, 16-byte aligned; its previous contents
// do not matter, the row-dot pass clears it).  `timed` records the events set
// by fa_set_backward_events around the main dK/dV kernel.
fa_status enqueue_backward(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dO, void* dq, void* dk, void* dv,
                           const AttnShape& s, float* Dbuf, float* acc, bool deterministic,
                           bool timed, cudaStream_t stream);

// The device address of a __device__ variable on the current device, looked
// up with cudaGetSymbolAddress once per device and cached (the host-side name
// of such a variable is a stand-in, never the device memory).  The cache has
// one slot per device the process sees.  nullptr if a CUDA call fails.
template <typename T>
void* symbol_address_cached(const T& symbol) {
  static std::mutex mu;
  static std::vector<void*> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (cache.empty()) {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || n < 1) return nullptr;
    cache.assign(static_cast<size_t>(n), nullptr);
  }
  if (static_cast<size_t>(dev) >= cache.size()) return nullptr;
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) return nullptr;
    cache[dev] = p;
  }
  return cache[dev];
}

// The forward at d = 128 on a pair of CTAs (fa_fwd_pair.cu): four query
// tiles per pair, products issued once for both CTAs.  tk must have 64 x 64
// boxes (half a key tile), tq and tv the usual 64 x 128 boxes.
cudaError_t launch_forward_pair(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, void* o, float* lse, const AttnShape& s,
                                uint32_t* err, cudaStream_t stream);
// Whether fa_forward / fa_forward_ex run shape s on a pair of CTAs.
bool forward_uses_pair(const AttnShape& s);

// Query rows per K/V-sharing unit of the forward: 0 = chosen per shape, 128,
// 256, or 512 (a pair of CTAs; d = 128).
void set_forward_rows_per_cta(int rows);
// Query rows per CTA (128 or 256) that the bf16 forward chooses for shape s
// on a GPU with `sms` multiprocessors when no setting forces one; host only.
int forward_rows_for(const AttnShape& s, int sms);
int forward_rows_per_cta();

// Backward pass kernels (see fa_bwd.cu).
// D = rowsum(dO o O) per row; if zero_acc is not null, also zeroes the fp32
// dQ accumulator [rows][d] (16-byte aligned).
cudaError_t launch_preprocess(const void* o, const void* dO, float* D, long long rows, int d,
                              cudaStream_t stream, float* zero_acc = nullptr);

struct BwdMaps {
  CUtensorMap q, k, v, dO;  // bf16, box 64 x 128 x 1 (k, v: 64 x 64 x 1 at d = 256), 128-byte swizzle
  CUtensorMap dq_acc;       // fp32 accumulator, box 32 x 128 x 1, 128-byte swizzle
  CUtensorMap dq_acc32;     // the same accumulator, box 32 x 32 x 1 (one warp's rows)
};

// Head dimension 64 (fa_bwd_d64.cu); launch_backward dispatches to it.
// with_dq = false: dK and dV only (the first kernel of the deterministic
// backward; dq_acc and the dq_acc map are not used).
cudaError_t launch_backward_d64(const BwdMaps& m, const float* lse, const float* D, void* dk,
                                void* dv, const AttnShape& s, uint32_t* err, cudaStream_t stream,
                                bool with_dq);

cudaError_t launch_backward(const BwdMaps& m, const float* lse, const float* D, float* dq_acc,
                            void* dk, void* dv, const AttnShape& s, uint32_t* err,
                            cudaStream_t stream, bool with_dq = true);

// dK and dV at head dimension 256 (fa_bwd_d256.cu): 64-key tiles, the
// accumulators held transposed; K/V maps with 64-row boxes.  dQ follows from
// launch_backward_dq.
cudaError_t launch_backward_d256_kv(const BwdMaps& m, const float* lse, const float* D, void* dk,
                                    void* dv, const AttnShape& s, uint32_t* err,
                                    cudaStream_t stream);

// dQ of the deterministic backward (fa_bwd_dq.cu): per query tile, key tiles
// in forward order, dq = bf16(scale * dS K) written directly, no atomics.
cudaError_t launch_backward_dq(const BwdMaps& m, const float* lse, const float* D, void* dq,
                               const AttnShape& s, uint32_t* err, cudaStream_t stream);

// Helpers defined in fa_api.cu for other translation units: the per-device
// error word the kernels' bounded waits report into, and tensor-map encoding
// for bf16 [planes][N][d] tensors and the fp32 dQ accumulator.
uint32_t* device_error_word();
bool encode_map_bf16(CUtensorMap* m, const void* ptr, int d, int N, long long planes);
bool encode_map_f32_acc(CUtensorMap* m, const void* ptr, int d, int N, long long planes);
bool encode_map_f32_acc32(CUtensorMap* m, const void* ptr, int d, int N, long long planes);

cudaError_t launch_dq_finalize(const float* dq_acc, void* dq, long long n, float scale,
                               cudaStream_t stream);

}  // namespace fa
