/*
 * fa.h - C ABI of the exact-attention library for NVIDIA GB300 (sm_103a).
 *
 * Exact scaled-dot-product attention,
 *     O = softmax(Q K^T * scale + causal mask) V,
 * computed tile by tile with the online softmax so that the N x N scores S and
 * weights P never reach device memory ("FlashAttention: l'attenzione che non
 * spreca memoria", sections "L'idea: lavorare a tessere, mai scrivere la
 * matrice" and "La online softmax, con i numeri"; "L'attention fusionnee",
 * section "Le softmax en ligne").
 *
 * Conventions shared by every entry point
 *   - Tensors are contiguous, row-major, laid out [B][H][N][d] (batch, head,
 *     position, head dimension), the (batch, heads, N, d_k) layout of the
 *     PyTorch call in "FlashAttention: l'attenzione che non spreca memoria",
 *     section "Cosa si guadagna (e cosa costa)".  Q, O, dO, dQ carry H_q heads;
 *     K, V, dK, dV carry H_kv heads.  Query head h reads key/value head
 *     h / (H_q / H_kv): contiguous groups, the QUERY_GROUP_SIZE of the CUDA
 *     Tile kernel signature ("Flash Attention ... NVIDIA CUDA Tile",
 *     section "Definiendo la interfaz del kernel").
 *   - q, k, v, o, dO, dq, dk, dv hold bf16 values (IEEE binary16 with an 8-bit
 *     exponent, "bfloat16"); lse holds fp32.  All arithmetic accumulates in
 *     fp32; outputs are rounded to bf16 once, round-to-nearest-even.
 *   - All pointers are DEVICE pointers on the current CUDA device.  The
 *     caller allocates and owns every buffer; the library never frees or
 *     retains them.  Each of q, k, v, o, dO, dq, dk, dv must be 16-byte
 *     aligned (tensor-memory-accelerator copies); lse 4-byte aligned.
 *   - causal = 1 applies the positional mask: query i sees keys j <= i
 *     ("Flash Attention ... NVIDIA CUDA Tile", section "Atencion causal":
 *     mask 0 where i >= j, -inf where i < j).  causal = 0: no mask.
 *   - scale multiplies Q K^T; it must be finite and > 0 (1/sqrt(d) is usual).
 *   - Work is enqueued on `stream` and the call returns without waiting.  A
 *     fault inside a kernel surfaces at the caller's next synchronisation;
 *     fa_last_device_error reports a timed-out wait inside a kernel.
 *   - Nothing is printed and nothing aborts.
 *
 * Supported sizes: d in {64, 96, 128, 256} (fa_forward_fp8: 128 only);
 * B, H_q, H_kv, N >= 1; H_q % H_kv == 0;
 * B * H_q * N * d < 2^40.
 */
#ifndef FA_H
#define FA_H

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, bad size, bad scale */
  FA_ERR_UNSUPPORTED = 2,      /* head dimension d not supported by the call */
  FA_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed */
  FA_ERR_DEVICE_TIMEOUT = 4    /* a bounded wait inside a kernel ran out */
} fa_status;

/*
 * Forward pass.  Source: "L'attention fusionnee", section "Le softmax en
 * ligne" (per key tile: m' = max(m, max s); p = exp(s - m');
 * l = l e^(m - m') + sum p; o = o e^(m - m') + p v; one division o / l at the
 * end) and section "La passe arriere : recalculer plutot que garder" (the forward
 * stores L = m + ln l).
 *
 *   q   [B][H_q][N][d]   bf16, read
 *   k   [B][H_kv][N][d]  bf16, read
 *   v   [B][H_kv][N][d]  bf16, read
 *   o   [B][H_q][N][d]   bf16, written: softmax(q k^T scale + mask) v
 *   lse [B][H_q][N]      fp32, written: natural log of sum_j exp(scale q.k_j)
 *                        over the keys the row sees (the scaled-score domain)
 *
 * Returns FA_OK once the work is enqueued; FA_ERR_INVALID_ARGUMENT or
 * FA_ERR_UNSUPPORTED before any launch; FA_ERR_CUDA if the launch failed.
 */
fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H_q, int H_kv, int N, int d, float scale, int causal,
                     cudaStream_t stream);

/*
 * Forward pass for queries that continue a longer key sequence (prefill
 * against keys already cached), following the position offset `input_pos` of
 * the CUDA Tile kernel signature ("Flash Attention ... NVIDIA CUDA Tile",
 * section "Definiendo la interfaz del kernel").  Query row i sits at absolute
 * position q_offset + i; with causal = 1 it sees keys j <= q_offset + i, with
 * causal = 0 every key.  fa_forward(..., N, ...) is fa_forward_ex with
 * N_q = N_kv = N and q_offset = 0.
 *
 *   q, o  [B][H_q][N_q][d]    bf16;   lse [B][H_q][N_q] fp32
 *   k, v  [B][H_kv][N_kv][d]  bf16
 *   q_offset >= 0 (every query row then sees at least key 0); N_q, N_kv >= 1.
 *
 * Same conventions and return codes as fa_forward.
 */
fa_status fa_forward_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H_q, int H_kv, int N_q, int N_kv, int d, float scale, int causal,
                        int q_offset, cudaStream_t stream);

/*
 * FP8 forward.  "FlashAttention: l'attenzione che non spreca memoria", section
 * on what comes next: the tensor cores gain narrower formats down to FP8
 * (8 bits), which halve again the bytes to move.  The same computation as
 * fa_forward with Q, K and V stored as e4m3 (OCP FP8, 4 exponent and 3
 * mantissa bits) times one fp32 factor per tensor, the products Q K^T and
 * P V on the FP8 tensor cores with fp32 accumulation, the softmax in fp32,
 * and P rounded to e4m3 (round to nearest even) for P V.
 *
 *   q    [B][H_q][N][d]   e4m3, read; its values are q * q_descale
 *   k    [B][H_kv][N][d]  e4m3, read; values k * k_descale
 *   v_t  [B][H_kv][d][N]  e4m3, read: V transposed (N contiguous), values
 *                         v_t * v_descale (every operand is then K-major)
 *   o    [B][H_q][N][d]   bf16, written;  lse [B][H_q][N] fp32, written
 *
 * d = 128 only (else FA_ERR_UNSUPPORTED); N a multiple of 16 (the rows of
 * v_t are N bytes long and must start 16 bytes apart); q_descale, k_descale,
 * v_descale finite and > 0.  Otherwise as fa_forward.
 */
fa_status fa_forward_fp8(const void* q, const void* k, const void* v_t, void* o, float* lse,
                         int B, int H_q, int H_kv, int N, int d, float scale, float q_descale,
                         float k_descale, float v_descale, int causal, cudaStream_t stream);

/*
 * Query rows per CTA of the bf16 forward (fa_forward, fa_forward_ex) at
 * d = 64, 96 and 128 — the B_r of the tiling in "FlashAttention:
 * l'attenzione che non spreca memoria", section "L'idea: lavorare a
 * tessere", chosen per problem size as the autotuning row of "Flash
 * Attention ... NVIDIA CUDA Tile", section "Resumen: La pila de
 * optimización", does per sequence length:
 *   0    chosen per shape (the default), as fa_forward_tile_rows_for says;
 *   128  one 128-row query tile per CTA;
 *   256  two 128-row query tiles per CTA sharing each K/V tile;
 *   512  at d = 128: a pair of CTAs (a cluster of two) with two query tiles
 *        each, whose tensor-core products are issued once for both CTAs
 *        (M = 256 across the pair) and which each load half of every K/V
 *        tile; at other d as 256.
 * All give the same results up to rounding order (256 and 512 the same
 * bits).  d = 256 always uses 128; fa_forward_fp8 always uses 256.
 * Process-wide; returns
 * FA_ERR_INVALID_ARGUMENT for any other value.
 */
fa_status fa_set_forward_tile_rows(int rows);

/*
 * The query rows per CTA (128 or 256) that fa_forward / fa_forward_ex choose
 * when fa_set_forward_tile_rows is 0, for a problem of those sizes (the
 * arguments of fa_forward_ex) on a GPU with `sms` multiprocessors.  Each
 * grid's finish time is estimated by list scheduling: its CTAs, in launch
 * order, each start on the multiprocessor that frees first, one CTA per
 * multiprocessor at a time, and cost a per-CTA overhead plus their key-tile
 * steps at costs fitted on GB300; the grid that finishes first is chosen
 * (d = 256 always 128).  Pure host computation: needs no GPU, enqueues
 * nothing.  Returns 0 for arguments fa_forward_ex would reject (and for
 * sms < 1).
 */
int fa_forward_tile_rows_for(int B, int H_q, int H_kv, int N_q, int N_kv, int d, int causal,
                             int q_offset, int sms);

/*
 * Backward pass.  Source: "L'attention fusionnee", section "La passe
 * arriere : recalculer plutot que garder": P is rebuilt tile by tile from the saved L as p = exp(s - L);
 *   dV = P^T dO;  dS = P o (dO V^T - D) with D = rowsum(dO o O);
 *   dQ = dS K scale;  dK = dS^T Q scale.
 * D is computed by a reduction kernel before everything else (same section).
 * For grouped-query attention, dK and dV of a shared head are the sums over
 * the query heads that read it.
 *
 *   q, k, v, o, lse  as produced for / by fa_forward with the same sizes
 *   dO  [B][H_q][N][d]   bf16, read: gradient of the loss w.r.t. o
 *   dq  [B][H_q][N][d]   bf16, written
 *   dk  [B][H_kv][N][d]  bf16, written
 *   dv  [B][H_kv][N][d]  bf16, written
 *
 * Scratch: B*H_q*N*4 bytes for D and B*H_q*N*d*4 bytes for an fp32 dQ
 * accumulator are taken stream-ordered (cudaMallocAsync on `stream`) and
 * released the same way before the call returns; the caller's buffers are
 * not used as scratch.  dq/dk/dv must not alias any input.
 *
 * At d = 256 the call runs the two kernels of fa_backward_deterministic (its
 * results are then bit-reproducible) and takes only D as scratch: the fp32
 * dK and dV of a 128-key tile would fill the whole tensor memory, so dK and
 * dV come from 64-key tiles with the accumulators held transposed, and dQ
 * from a kernel that owns query tiles.
 *
 * Returns as fa_forward; FA_ERR_CUDA also when the scratch allocation fails.
 */
fa_status fa_backward(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                      int H_q, int H_kv, int N, int d, float scale, int causal,
                      cudaStream_t stream);

/*
 * Backward pass whose results are bit-for-bit reproducible from run to run.
 * Source: "L'attention fusionnee", section "La passe arriere : recalculer
 * plutot que garder": instead of one kernel that adds each key tile's share
 * of dQ with atomic additions, one kernel computes dK and dV and a second
 * computes dQ, walking the key tiles in the forward pass's order; it redoes
 * three products but needs no atomics, so the result does not depend on the
 * order in which the GPU runs its blocks.
 *
 * Arguments, layouts, outputs and return codes are those of fa_backward.
 * Scratch: only D (B*H_q*N*4 bytes), taken and released stream-ordered.
 */
fa_status fa_backward_deterministic(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dO, void* dq, void* dk,
                                    void* dv, int B, int H_q, int H_kv, int N, int d, float scale,
                                    int causal, cudaStream_t stream);

/*
 * Scratch reserved by the library for fa_backward_noalloc, in bytes (32 MiB).
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * fa_backward without any device allocation (an addition of this library;
 * the source pages describe no such entry point).
 *
 * For callers that cannot allocate device memory at the point where they
 * run the backward pass: for example an application whose device memory is
 * already reserved by another allocator, or a plug-in that an inference or
 * training engine calls at enqueue time under a no-allocation rule.  The
 * arguments, layouts, results and return codes are those of fa_backward; the
 * results agree with fa_backward's within rounding (dQ is summed in fp32 in
 * an order that can differ between runs).
 *
 * Instead of the memory pool it uses a fixed array of FA_NOALLOC_SCRATCH_BYTES
 * inside the library, reserved on every GPU that loads the library until the
 * process exits.  It holds D and the fp32 dQ accumulator, so a call needs
 *     ceil(B*H_q*N*4 / 1024)*1024 + B*H_q*N*d*4  bytes
 * (for example B=2, H_q=8, N=4096, d=64: about 16.3 MiB), or B*H_q*N*4 bytes
 * at d = 256, where the backward has no accumulator; larger problems are
 * rejected with FA_ERR_INVALID_ARGUMENT before anything is launched.
 *
 * The array is shared by all calls on a device and keeps the last call's
 * contents; each call clears the part that must start at zero.  Calls whose
 * work overlaps on the GPU (on different streams, or from several threads)
 * race on that array: serialise them, e.g. by issuing them on one stream.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture begins.  No cudaMalloc, cudaFree or other
 * allocating routine is called.
 */
fa_status fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dO, void* dq, void* dk, void* dv,
                              int B, int H_q, int H_kv, int N, int d, float scale, int causal,
                              cudaStream_t stream);

/*
 * The backward pass's first step on its own: D[r] = sum_c dO[r][c] * O[r][c]
 * for every row r of [rows][d] bf16 matrices, accumulated in fp32 ("L'attention
 * fusionnee", section "La passe arriere : recalculer plutot que garder": the sum of dP x P over a row of P
 * equals the sum of dO x O over the row, one value per row).
 *
 *   o, dO  [rows][d] bf16 device pointers, 16-byte aligned, read
 *   D      [rows]    fp32 device pointer, written
 * d in {64, 96, 128, 256}; rows >= 1.  Same return codes as fa_forward.
 */
fa_status fa_backward_preprocess(const void* o, const void* dO, float* D, long long rows, int d,
                                 cudaStream_t stream);

/* Static, NUL-terminated description of a status code. */
const char* fa_status_string(fa_status s);

/*
 * Synchronises `stream`, then reports what the kernels left behind: FA_ERR_CUDA
 * for a pending CUDA error, FA_ERR_DEVICE_TIMEOUT if a bounded wait inside a
 * kernel of this library ran out since the last call (the flag is then
 * cleared), FA_OK otherwise.  Every wait inside the kernels gives up after
 * about a second instead of hanging; the kernel then skips its remaining work.
 */
fa_status fa_last_device_error(cudaStream_t stream);

/*
 * Diagnostics for the bounded-wait error path (the pages have no counterpart):
 * launches one thread that waits on a barrier nothing completes, gives up
 * after `limit_ms` milliseconds (1..2000) and records a timeout exactly as the
 * attention kernels do, so that a caller can check that fa_last_device_error
 * reports FA_ERR_DEVICE_TIMEOUT and that the device stays usable.  Returns
 * FA_OK once enqueued, FA_ERR_INVALID_ARGUMENT for a limit out of range.
 */
fa_status fa_selftest_wait_timeout(int limit_ms, cudaStream_t stream);

/*
 * Timing hook for the backward pass's main kernel (diagnostics; the pages have
 * no counterpart).  When both events are non-NULL, every later fa_backward
 * call records `before` on its stream immediately before launching the main
 * dK/dV/dQ kernel and `after` immediately after it, so a caller can time that
 * kernel alone with cudaEventElapsedTime.  Pass NULL, NULL to switch it off.
 * The events are owned by the caller and must outlive their use.  The setting
 * is process-wide and not synchronised: set it from one thread.
 */
void fa_set_backward_events(cudaEvent_t before, cudaEvent_t after);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
