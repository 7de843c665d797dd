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

}  // namespace

extern "C" fa_status fa_backward_noalloc(const void* q, const void* k, const void* v,
                                         const void* o, const float* lse, const void* dO,
                                         void* dq, void* dk, void* dv, int B, int H_q, int H_kv,
                                         int N, int d, float scale, int causal,
                                         cudaStream_t stream) {
  // The checks of fa_backward, in the same order, so both return the same codes.
  const fa_status st = fa::validate_backward(q, k, v, o, lse, dO, dq, dk, dv, B, H_q, H_kv, N, d,
                                             scale, causal);
  if (st != FA_OK) return st;
  // The scratch must hold what fa_backward would take from the pool: D for
  // every query row and, unless d = 256 (two kernels, no accumulator), the
  // fp32 dQ accumulator.  validate() bounds B*H_q*N*d below 2^40, so the
  // sizes cannot overflow.
  size_t acc_off = 0;
  const size_t need = fa::backward_scratch_bytes(B, H_q, N, d, false, &acc_off);
  if (need > static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES)) return FA_ERR_INVALID_ARGUMENT;
  void* base = scratch_address();
  if (!base) return FA_ERR_CUDA;
  float* Dbuf = static_cast<float*>(base);
  float* acc = acc_off ? reinterpret_cast<float*>(static_cast<char*>(base) + acc_off) : nullptr;
  fa::AttnShape s{B, H_q, H_kv, N, d, scale, causal};
  // The accumulator keeps the previous call's sums: the row-dot pass clears it.
  return fa::enqueue_backward(q, k, v, o, lse, dO, dq, dk, dv, s, Dbuf, acc,
                              /*deterministic=*/false, /*timed=*/false, stream);
}
