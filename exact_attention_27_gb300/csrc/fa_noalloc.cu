// fa_backward_noalloc: the backward pass without any device allocation.
//
// fa_backward takes its scratch (the per-row D vector and the fp32 dQ
// accumulator) from the stream-ordered memory pool on every call.  Some
// callers cannot do that: an application whose device memory is already
// reserved by another allocator (a framework's caching allocator, a static
// memory plan in an inference runtime) may see that allocation fail, and an
// engine that hands work to a plug-in at enqueue time may forbid allocation
// there altogether.  This entry point serves them: its scratch is the
// fixed-size array below, which is part of the library's device image and is
// reserved on every GPU that loads the library, until the process exits.
//
// The kernels are the same ones fa_backward launches; only where the scratch
// comes from differs.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

// Scratch of fa_backward_noalloc: D (fp32 per query row, padded to 1 KiB)
// followed by the fp32 dQ accumulator.  Shared by every call on a device.
static __device__ __align__(256) unsigned char fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Device address of fa_noalloc_scratch on the current device, looked up once
// per device.  In host code the array's name stands for a host-side shadow,
// never for the device memory itself, so kernels must be given this address.
void* scratch_address() { return fa::symbol_address_cached(fa_noalloc_scratch); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" fa_status fa_backward_noalloc(const void* q, const void* k, const void* v,
                                         const void* o, const float* lse, const void* dO,
                                         void* dq, void* dk, void* dv, int B, int H_q, int H_kv,
                                         int N, int d, float scale, int causal,
                                         cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARGUMENT;
  // The checks of fa_backward, in the same order, so both return the same codes.
  const fa_status st = fa::validate(B, H_q, H_kv, N, d, scale, causal);
  if (st != FA_OK) return st;
  if (d == 256) return FA_ERR_UNSUPPORTED;
  const void* p16[] = {q, k, v, o, dO, dq, dk, dv};
  for (const void* p : p16)
    if (!aligned16(p)) return FA_ERR_INVALID_ARGUMENT;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_INVALID_ARGUMENT;

  // The scratch must hold D and the accumulator for every query row.
  const double rows_d = static_cast<double>(B) * H_q * N;
  const double need = std::ceil(rows_d * 4.0 / 1024.0) * 1024.0 + rows_d * d * 4.0;
  if (need > static_cast<double>(FA_NOALLOC_SCRATCH_BYTES)) return FA_ERR_INVALID_ARGUMENT;
  const long long rows = static_cast<long long>(B) * H_q * N;
  const size_t acc_off = (static_cast<size_t>(rows) * 4 + 1023) & ~static_cast<size_t>(1023);

  void* base = scratch_address();
  uint32_t* err = fa::device_error_word();
  if (!base || !err) return FA_ERR_CUDA;
  float* Dbuf = static_cast<float*>(base);
  float* acc = reinterpret_cast<float*>(static_cast<char*>(base) + acc_off);

  fa::BwdMaps m;
  const bool ok = fa::encode_map_bf16(&m.q, q, d, N, static_cast<long long>(B) * H_q) &&
                  fa::encode_map_bf16(&m.k, k, d, N, static_cast<long long>(B) * H_kv) &&
                  fa::encode_map_bf16(&m.v, v, d, N, static_cast<long long>(B) * H_kv) &&
                  fa::encode_map_bf16(&m.dO, dO, d, N, static_cast<long long>(B) * H_q) &&
                  fa::encode_map_f32_acc(&m.dq_acc, acc, d, N, static_cast<long long>(B) * H_q) &&
                  fa::encode_map_f32_acc32(&m.dq_acc32, acc, d, N, static_cast<long long>(B) * H_q);
  if (!ok) return FA_ERR_CUDA;
  fa::AttnShape s{B, H_q, H_kv, N, d, scale, causal};
  // The accumulator keeps the previous call's sums: the preprocess clears it.
  cudaError_t e = fa::launch_preprocess(o, dO, Dbuf, rows, d, stream, acc);
  if (e == cudaSuccess) e = fa::launch_backward(m, lse, Dbuf, acc, dk, dv, s, err, stream);
  if (e == cudaSuccess) e = fa::launch_dq_finalize(acc, dq, rows * d, scale, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
