// Forward pass of exact attention on sm_103a.
//
// One CTA owns one tile of 128 query rows of one (batch, query head) and
// streams the key/value tiles of its key/value head past it ("FlashAttention:
// l'attenzione che non spreca memoria", section "L'idea: lavorare a tessere,
// mai scrivere la matrice": the query block stays, K_j / V_j blocks move, the
// S_ij tile is B_r x B_c, here 128 x 128).
//
// Each CTA owns two consecutive query tiles (A and B) and keeps one softmax
// warpgroup per tile, so that one tile's softmax runs while the tensor core
// works on the other tile's products (a ping-pong between the two).
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: thread t owns
//              query row t of its tile.  Online softmax per key tile, rescale
//              of the O accumulator, epilogue.
//   warp 8     TMA producer: both Q tiles once, then K_j and V_j into a ring.
//   warps 10-11 idle (they complete the third warpgroup)
//   warp 9     MMA issuer (one thread) and TMEM owner, in the order
//              S_A(0) S_B(0), then per key tile j:
//              O_A += P_A V_j, S_A(j+1) = Q_A K_{j+1}^T, O_B += P_B V_j, S_B(j+1)
//              (S: A and B from shared memory; O: A = P from tensor memory);
//              at D = 64: S_A(0) S_B(0) S_A(1), then per key tile j:
//              O_A += P_A V_j, S_B(j+1), O_B += P_B V_j, S_A(j+2).
// Registers: launched at 168 per thread; the third warpgroup gives most of
// its share to the two softmax warpgroups (56 / 224 / 224: 128 x (224 + 224
// + 56) = 384 x 168, the launch total).
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   columns   0..127  S of tile A    (P as packed bf16 overwrites columns 0..63)
//   columns 128..255  S of tile B
//   columns 256..256+2DP-1  O accumulators of tiles A and B (fp32; DP = D
//              rounded up to a multiple of 64)
// except at D = 64, where three S buffers (columns 0..383) rotate between
// the two tiles and O_A, O_B sit at 384 and 448: a tile's next S is then
// computed while its softmax still works on the current one.
//
// Online softmax ("L'attention fusionnee", section "Le softmax en ligne"):
// per key tile m' = max(m, max s), p = exp(s - m'), l = l e^(m - m') + sum p,
// o = o e^(m - m') + p v, one division o / l after the last tile.  It runs in
// the base-2 domain with scale * log2(e) folded into one multiply-add (the
// exp2 form of "Flash Attention ... NVIDIA CUDA Tile", kernel interface
// section).  The reference point m is moved only when the running maximum has
// grown by more than kRescaleThreshold (in log2 units); otherwise the old m is
// kept for both o and l, which leaves o / l unchanged and bounds every p by
// 2^kRescaleThreshold.  The rescale of O then happens on few tiles.
//
// Causal masking ("L'attention fusionnee", same section: tiles that lie wholly
// in the future are never visited; the mask is positional, no mask tensor):
// query row i sits at absolute position q_offset + i (the input_pos of the
// CUDA Tile kernel; 0 when queries and keys are the same sequence) and sees
// keys j <= q_offset + i, so a query tile visits key tiles up to the one
// holding its last row's position, and only tiles crossing the diagonal are
// masked.  Keys at or past Nk (ragged tail) are masked too.
//
// Every mbarrier wait is bounded (about a second); on expiry the kernel sets
// an error bit, every role skips its remaining work and the CTA exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <atomic>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <vector>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

// Head dimension D in {64, 96, 128}.  Tiles are stored DP = D rounded up to
// a multiple of 64 columns wide (whole 128-byte swizzle atoms); for D = 96
// the copies fill columns 96..127 with zeros (they lie outside the tensor),
// Q K^T runs over the D real columns only, and P V runs at N = D (a
// multiple of 16, as the MMA allows), so no O column past D is computed.
//
// FP8 = true: Q, K and V^T are e4m3 (one byte per element, D = 128: one
// 128-byte row per tile row, so SUB = 1), the products run as kind::f8f6f4,
// P is rounded to e4m3 (4 per TMEM column) and V comes transposed ([d][N]),
// so that both operands of O += P V are K-major.
template <int D, bool FP8 = false>
struct FwdCfg {
  static constexpr int DP = (D + 63) / 64 * 64;  // padded head dimension
  static constexpr int BM = 128;                 // query rows per tile (MMA M)
  static constexpr int BN = 128;                 // keys per tile (MMA N of Q K^T)
  static constexpr int SUB = FP8 ? 1 : DP / 64;  // 128-byte column blocks per row
  static constexpr int SUB_BYTES = 128 * 128;    // one 128-row x 128-byte block
  static constexpr int TILE = SUB * SUB_BYTES;   // one 128 x D tile
  static constexpr int NS = (D == 64 || FP8) ? 4 : 2;  // K/V ring stages
  static constexpr int OFF_Q = 0;                // two query tiles
  static constexpr int OFF_K = OFF_Q + 2 * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_BAR = OFF_V + NS * TILE;
  // barrier slots
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;
  static constexpr int B_KEMPTY = B_KFULL + NS;
  static constexpr int B_VFULL = B_KEMPTY + NS;
  static constexpr int B_VEMPTY = B_VFULL + NS;
  // At DP = 64 three S buffers of 128 columns rotate between the two tiles
  // (the n-th S issued goes to buffer n % 3; P overwrites the first 64
  // columns of its own S), which with the two O accumulators fills the 512
  // columns; the MMA issuer's order makes each reuse safe.  Otherwise each
  // tile has its own S columns.
  static constexpr bool ROT3 = (DP == 64) && !FP8;
  static constexpr int NSB = ROT3 ? 3 : 2;       // S buffers
  static constexpr int B_SFULL = B_VEMPTY + NS;  // [NSB] S in buffer (ROT3) or of tile x
  // P written over the S of buffer b (4 warp arrivals).  With ROT3 a tile's
  // softmax may finish two steps before the MMA issuer waits for the first
  // of them (say while it waits for a late V tile), so the barrier is per
  // buffer: the buffer's next P needs an S issued after this P's P V, and
  // the barrier is never two phases ahead of the issuer.  Without ROT3 a
  // tile's next S follows its own P V, and buffer x is tile x's.
  static constexpr int B_PFULL = B_SFULL + NSB;  // [NSB]
  static constexpr int B_ODONE = B_PFULL + NSB;  // [2] per query tile: O += P V done
  static constexpr int B_OFIN = B_ODONE + 2;     // [2] per query tile, once: its last P V done
  static constexpr int B_DRAIN = B_OFIN + 2;     // abort path: MMAs in flight
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;  // tmem slot, abort word
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = ROT3 ? 384 : 256;  // O of tile x at COL_O + x * DP
};

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  int N;         // query rows
  int Nk;        // key/value rows
  int q_offset;  // absolute position of query row 0
  int Hq;
  int G;          // query heads per key/value head
  int n_qtiles;
  int n_qpairs;   // CTAs per head: two query tiles each
  int n_ktiles;
  int n_heads;          // B * Hq
  int heads_per_group;  // launch-order grouping, a multiple of G
  float scale_log2;  // scale * log2(e) (times the Q and K descales for FP8)
  float o_scale;     // factor on O in the epilogue (the V descale for FP8, else 1)
  uint32_t* err;
};

template <int D, bool CAUSAL, bool FP8 = false>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  // Launch order: heads are taken in groups of p.heads_per_group (sized on
  // the host so that the group's K/V fits comfortably in L2); within a group
  // the heaviest causal query-tile pairs of all its heads come first.
  const int per_group = p.heads_per_group * p.n_qpairs;
  const int grp = static_cast<int>(blockIdx.x) / per_group;
  const int rem = static_cast<int>(blockIdx.x) - grp * per_group;
  const int in_grp = min(p.heads_per_group, p.n_heads - grp * p.heads_per_group);
  const int pi_ = rem / in_grp;
  const int bh = grp * p.heads_per_group + (rem - pi_ * in_grp);  // flattened (batch, query head)
  const int pair = CAUSAL ? (p.n_qpairs - 1 - pi_) : pi_;
  const int b = bh / p.Hq;
  const int hq = bh - b * p.Hq;
  const int kvz = b * (p.Hq / p.G) + hq / p.G;  // flattened (batch, kv head)
  // Key tiles visited by query tile 2*pair + x (0 if that tile is past N).
  auto tiles_for = [&](int x) -> int {
    const int qt = 2 * pair + x;
    if (qt >= p.n_qtiles) return 0;
    return CAUSAL ? min((p.q_offset + qt * C::BM + C::BM - 1) / C::BN + 1, p.n_ktiles)
                  : p.n_ktiles;
  };
  const int nA = tiles_for(0);
  const int nB = tiles_for(1);
  const int n_kv = max(nA, nB);

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_QFULL), 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 1);
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int x = 0; x < C::NSB; ++x) {
      mbar_init(bar(C::B_SFULL + x), 1);
      mbar_init(bar(C::B_PFULL + x), 4);  // one arrival per softmax warp of the tile
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::B_ODONE + x), 1);
      mbar_init(bar(C::B_OFIN + x), 1);
    }
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched as a programmatic dependent of the grid before it in the
  // stream: Q, K and V are read, and O and L written, only once that grid
  // has completed; the grid after this one may be scheduled from then on.
  grid_dependency_wait();
  grid_launch_dependents();

  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t sK = sbase + C::OFF_K;
  const uint32_t sV = sbase + C::OFF_V;

  if (warp >= 8) {
  reg_decrease<56>();
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t keep = policy_evict_last();  // K/V are re-read by the other query tiles
      mbar_arrive_expect_tx(bar(C::B_QFULL), 2 * C::TILE);
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int s = 0; s < C::SUB; ++s)
          tma_load_3d(sQ + x * C::TILE + s * C::SUB_BYTES, &tmQ, bar(C::B_QFULL), 64 * s,
                      (2 * pair + x) * C::BM, bh);
      int issued = 0;  // K/V tiles whose loads were issued
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % C::NS;
        const uint32_t ph = ((j / C::NS) - 1) & 1;
        if (j >= C::NS &&
            !mbar_wait(bar(C::B_KEMPTY + st), ph, abort_flag, p.err, kErrTimeoutLoad))
          break;
        mbar_arrive_expect_tx(bar(C::B_KFULL + st), C::TILE);
#pragma unroll
        for (int s = 0; s < C::SUB; ++s)
          tma_load_3d_hint(sK + st * C::TILE + s * C::SUB_BYTES, &tmK, bar(C::B_KFULL + st),
                           64 * s, j * C::BN, kvz, keep);
        if (j >= C::NS &&
            !mbar_wait(bar(C::B_VEMPTY + st), ph, abort_flag, p.err, kErrTimeoutLoad))
          break;
        mbar_arrive_expect_tx(bar(C::B_VFULL + st), C::TILE);
        if constexpr (FP8) {
          // V^T: 128 rows of d, each 128 keys (bytes) long.
          tma_load_3d_hint(sV + st * C::TILE, &tmV, bar(C::B_VFULL + st), j * C::BN, 0, kvz,
                           keep);
        } else {
#pragma unroll
          for (int s = 0; s < C::SUB; ++s)
            tma_load_3d_hint(sV + st * C::TILE + s * C::SUB_BYTES, &tmV, bar(C::B_VFULL + st),
                             64 * s, j * C::BN, kvz, keep);
        }
        issued = j + 1;
      }
      if (*abort_flag) {
        // Let the copies already issued land before the CTA's memory is released.
        mbar_wait_timed(bar(C::B_QFULL), 0);
        for (int j = max(0, issued - C::NS); j < issued; ++j) {
          mbar_wait_timed(bar(C::B_KFULL + j % C::NS), (j / C::NS) & 1);
          mbar_wait_timed(bar(C::B_VFULL + j % C::NS), (j / C::NS) & 1);
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // Order: S_A(0) S_B(0), then per key tile j: PV_A(j) S_A(j+1) PV_B(j)
    // S_B(j+1), so that each tile's softmax overlaps the other tile's MMAs.
    if (elect_one()) {
      constexpr uint32_t ID_S =
          FP8 ? idesc_e4m3_f32(128, 128) : idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t ID_O =
          FP8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(128, D, false, true);
      const uint64_t q_desc = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t k_desc = smem_desc_sw128(sK, 16, 1024);
      // bf16: V is [keys][d], read MN-major; FP8: V^T is [d][keys], read K-major.
      const uint64_t v_desc = smem_desc_sw128(sV, FP8 ? 16 : C::SUB_BYTES, 1024);
      const int nx[2] = {nA, nB};
      bool ok = mbar_wait(bar(C::B_QFULL), 0, abort_flag, p.err, kErrTimeoutMma);
      // S_x(j) = Q_x K_j^T into S buffer `buf`.
      auto issue_s = [&](int x, int j, int buf) {
        const uint32_t d_tmem = tmem + buf * 128;
        const uint64_t qd = desc_add(q_desc, x * C::TILE);
        const uint64_t kd = desc_add(k_desc, (j % C::NS) * C::TILE);
        if constexpr (FP8) {
          // 32 e4m3 elements (32 bytes) of d per step.
          mma_ss_f8_k<ID_S, 0>(d_tmem, qd, kd);
#pragma unroll
          for (int kk = 1; kk < D / 32; ++kk)
            mma_ss_f8_k<ID_S, 1>(d_tmem, desc_add(qd, kk * 32), desc_add(kd, kk * 32));
        } else {
          mma_ss_k<ID_S, 0>(d_tmem, qd, kd);
#pragma unroll
          for (int kk = 1; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::SUB_BYTES + (kk & 3) * 32;
            mma_ss_k<ID_S, 1>(d_tmem, desc_add(qd, off), desc_add(kd, off));
          }
        }
        mma_commit(bar(C::B_SFULL + buf));
      };
      // K_j is used by the S products of both tiles; wait for it once and
      // release it after its last use.
      auto issue_s_both = [&](int j) -> bool {
        const int st = j % C::NS;
        if (!mbar_wait(bar(C::B_KFULL + st), (j / C::NS) & 1, abort_flag, p.err, kErrTimeoutMma))
          return false;
        tc_fence_after();
        return true;
      };
      if (!C::ROT3 && ok && n_kv > 0) {
        ok = issue_s_both(0);
        if (ok) {
          if (nA > 0) issue_s(0, 0, 0);
          if (nB > 0) issue_s(1, 0, 1);
          mma_commit(bar(C::B_KEMPTY + 0));
        }
      }
      if constexpr (C::ROT3) {
        // Three S buffers rotate between the tiles.  S issue order is A0 B0
        // A1 B1 ..., so S_x(j) is the n-th S issued, n = min(j + x, nA) +
        // min(j, nB), and goes to buffer n % 3.  Order: S_A(0) S_B(0) S_A(1),
        // then per key tile j: O_A += P_A V_j, S_B(j+1), O_B += P_B V_j,
        // S_A(j+2).  Each S then follows the P V of the S that held its buffer
        // before (number n - 3), and the tensor pipe runs in issue order, so
        // that P is read before it is overwritten; the softmax of a tile finds
        // its next S computed while it works on the current one.
        auto snum = [&](int x, int j) { return min(j + x, nA) + min(j, nB); };
        auto sbuf = [&](int x, int j) { return snum(x, j) % 3; };
        int k_waited = 0;  // K tiles waited for (first uses come in order)
        auto s3 = [&](int x, int j) -> bool {
          if (j >= k_waited) {
            if (!issue_s_both(j)) return false;
            k_waited = j + 1;
          }
          issue_s(x, j, sbuf(x, j));
          if (x == 1 || j >= nB) mma_commit(bar(C::B_KEMPTY + j % C::NS));  // K_j's last use
          return true;
        };
        auto pv3 = [&](int x, int j) -> bool {
          const int st = j % C::NS;
          if ((x == 0 || j >= nA) &&
              !mbar_wait(bar(C::B_VFULL + st), (j / C::NS) & 1, abort_flag, p.err, kErrTimeoutMma))
            return false;
          if (!mbar_wait(bar(C::B_PFULL + sbuf(x, j)), (snum(x, j) / 3) & 1, abort_flag, p.err,
                         kErrTimeoutMma))
            return false;
          tc_fence_after();
          const uint64_t vd = desc_add(v_desc, st * C::TILE);
          const uint32_t pa = tmem + sbuf(x, j) * 128;  // P packed over its S
          const uint32_t od = tmem + C::COL_O + x * C::DP;
          if (j == 0)
            mma_ts_k<ID_O, 0>(od, pa, vd);
          else
            mma_ts_k<ID_O, 1>(od, pa, vd);
#pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            mma_ts_k<ID_O, 1>(od, pa + kk * 8, desc_add(vd, kk * 2048));
          mma_commit(bar(C::B_ODONE + x));
          if (j == nx[x] - 1) mma_commit(bar(C::B_OFIN + x));
          if (x == 1 || j >= nB) mma_commit(bar(C::B_VEMPTY + st));  // V_j's last use
          return true;
        };
        if (ok && nA > 0) ok = s3(0, 0);
        if (ok && nB > 0) ok = s3(1, 0);
        if (ok && nA > 1) ok = s3(0, 1);
        for (int j = 0; ok && j < n_kv; ++j) {
          if (j < nA && !(ok = pv3(0, j))) break;
          if (j + 1 < nB && !(ok = s3(1, j + 1))) break;
          if (j < nB && !(ok = pv3(1, j))) break;
          if (j + 2 < nA && !(ok = s3(0, j + 2))) break;
        }
      }
      for (int j = 0; !C::ROT3 && ok && j < n_kv; ++j) {
        const int st = j % C::NS;
        if (!mbar_wait(bar(C::B_VFULL + st), (j / C::NS) & 1, abort_flag, p.err, kErrTimeoutMma))
          break;
        const bool next = (j + 1 < n_kv);
        bool k_ready = false;
#pragma unroll 1
        for (int x = 0; x < 2; ++x) {
          if (j >= nx[x]) continue;
          if (!mbar_wait(bar(C::B_PFULL + x), j & 1, abort_flag, p.err, kErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // O_x += P_x V_j: P packed over the first columns of tile x's S
          // (bf16: 16 keys = 8 columns per step; e4m3: 32 keys = 8 columns).
          const uint64_t vd = desc_add(v_desc, st * C::TILE);
          const uint32_t pa = tmem + x * 128;
          const uint32_t od = tmem + C::COL_O + x * C::DP;
          if constexpr (FP8) {
            if (j == 0)
              mma_ts_f8_k<ID_O, 0>(od, pa, vd);
            else
              mma_ts_f8_k<ID_O, 1>(od, pa, vd);
#pragma unroll
            for (int kk = 1; kk < 4; ++kk)
              mma_ts_f8_k<ID_O, 1>(od, pa + kk * 8, desc_add(vd, kk * 32));
          } else {
            if (j == 0)
              mma_ts_k<ID_O, 0>(od, pa, vd);
            else
              mma_ts_k<ID_O, 1>(od, pa, vd);
#pragma unroll
            for (int kk = 1; kk < 8; ++kk)
              mma_ts_k<ID_O, 1>(od, pa + kk * 8, desc_add(vd, kk * 2048));
          }
          mma_commit(bar(C::B_ODONE + x));
          if (next && j + 1 < nx[x]) {
            if (!k_ready) {
              if (!issue_s_both(j + 1)) {
                ok = false;
                break;
              }
              k_ready = true;
            }
            issue_s(x, j + 1, x);
          }
        }
        if (!ok) break;
        mma_commit(bar(C::B_VEMPTY + st));
        if (k_ready) mma_commit(bar(C::B_KEMPTY + (j + 1) % C::NS));
      }
      if (*abort_flag) {
        // Let the MMAs already issued finish before tensor memory is released.
        mma_commit(bar(C::B_DRAIN));
        mbar_wait_timed(bar(C::B_DRAIN), 0);
      }
    }
  }
  } else {
    reg_increase<224>();
    // ------------------------------------------------------------ softmax (rows)
    const int x = warp >> 2;            // query tile of this warpgroup
    const int row = threadIdx.x & 127;  // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int qt = 2 * pair + x;
    const int qi = qt * C::BM + row;
    const int nt = x == 0 ? nA : nB;
    const uint32_t col_o = C::COL_O + x * C::DP;
    const float c = p.scale_log2;
    float m_used = -INFINITY;  // reference maximum, log2 domain
    float l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      // Waits are made warp-uniform: the TMEM loads and stores below are
      // warp-collective, so either every lane goes on or every lane stops.
      // S_x(j): with ROT3 the n-th S issued, in buffer n % 3 (its (n / 3)-th
      // use); otherwise tile x's own columns.  P is stored over it as bf16
      // (e4m3 for FP8).
      const int sn = C::ROT3 ? min(j + x, nA) + min(j, nB) : 0;
      const int sb = C::ROT3 ? sn % 3 : x;
      const uint32_t col_s = sb * 128;
      const uint32_t col_p = col_s;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SFULL + sb), C::ROT3 ? (sn / 3) & 1 : j & 1,
                                             abort_flag, p.err, kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      // The row's 128 scores: four loads in flight, one wait.
      float s[128];
      {
        uint32_t r[128];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          tmem_ld32(tmem + lane_off + col_s + q4 * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(&r[q4 * 32]));
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < 128; ++t) s[t] = __uint_as_float(r[t]);
      }
      const int kbase = j * C::BN;
      const int qpos = p.q_offset + qi;  // absolute position of this row
      const bool need_mask =
          (kbase + C::BN > p.Nk) || (CAUSAL && kbase + C::BN - 1 > p.q_offset + qt * C::BM);
      if (need_mask) {
#pragma unroll
        for (int t = 0; t < 128; ++t) {
          const int key = kbase + t;
          if (key >= p.Nk || (CAUSAL && key > qpos)) s[t] = -INFINITY;
        }
      }
      // Row max over 8 independent partial maxima (a tree, not a 128-long
      // chain), two new values per three-input max.
      float pm[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) pm[u] = fmaxf(s[u], s[u + 8]);
#pragma unroll
      for (int t = 16; t < 128; t += 16)
#pragma unroll
        for (int u = 0; u < 8; ++u) pm[u] = fmax3(pm[u], s[t + u], s[t + u + 8]);
      const float mx = fmaxf(fmax3(pm[0], pm[1], pm[2]),
                             fmaxf(fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      const float m_new = fmaxf(m_used, mx * c);
      float alpha = 1.0f;
      const bool upd = m_new > m_used + kRescaleThreshold;
      if (upd) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
      }
      const float m_ref = (m_used == -INFINITY) ? 0.0f : m_used;
      // exp2(s c - m) with the multiply-add on pairs; 4 independent packed sums.
      const uint64_t c2 = f2_pack(c, c);
      const uint64_t nm2 = f2_pack(-m_ref, -m_ref);
      uint64_t ps2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) ps2[u] = 0ull;
      if constexpr (FP8) {
        // P rounded to e4m3, four keys per TMEM column (the lowest key in the
        // lowest byte); the running sum uses the fp32 values.
        uint32_t pk8[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(s[4 * t], s[4 * t + 1]), c2, nm2), x0, x1);
          f2_unpack(f2_fma(f2_pack(s[4 * t + 2], s[4 * t + 3]), c2, nm2), x2, x3);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
          ps2[(2 * t) & 3] = f2_add(ps2[(2 * t) & 3], f2_pack(p0, p1));
          ps2[(2 * t + 1) & 3] = f2_add(ps2[(2 * t + 1) & 3], f2_pack(p2, p3));
          pk8[t] = pack_e4m3x4(p0, p1, p2, p3);
        }
        tmem_st32(tmem + lane_off + col_p, pk8);
      } else {
        uint32_t pk[64];
  #pragma unroll
        for (int t = 0; t < 64; ++t) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(s[2 * t], s[2 * t + 1]), c2, nm2), x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          ps2[t & 3] = f2_add(ps2[t & 3], f2_pack(p0, p1));
          pk[t] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tmem + lane_off + col_p, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(tmem + lane_off + col_p + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      }
      float sum, sum_hi;
      f2_unpack(f2_add(f2_add(ps2[0], ps2[1]), f2_add(ps2[2], ps2[3])), sum, sum_hi);
      sum += sum_hi;
      l = l * alpha + sum;
      // O holds P_0..P_{j-1} contributions; it must be final before it is
      // rescaled.  The S just waited for was issued, by the same thread,
      // after the P V that read its buffer before (without ROT3, O += P_x(j-1)
      // V), and a commit tracks every earlier tcgen05 operation of its
      // thread, so that product has completed and P_x(j) may overwrite the
      // columns it read.  The wait below is for the rescale: without ROT3 it
      // returns at once; with ROT3 the S implies only O += P_x(j-2) V, and it
      // waits for O += P_x(j-1) V.  Either way the barrier has completed the
      // phase before the one waited for, and O += P_x(j) V waits for this
      // tile's P, so it is never two phases from the waiter.
      const bool resc = j > 0 && __any_sync(0xffffffffu, upd);
      if (resc) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_ODONE + x), (j - 1) & 1, abort_flag,
                                               p.err, kErrTimeoutSoftmax));
        if (!ok) break;
      }
      if (resc) {
        tc_fence_after();
#pragma unroll
        for (int q4 = 0; q4 < D / 32; ++q4) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + col_o + q4 * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 32; ++t) r[t] = __float_as_uint(__uint_as_float(r[t]) * alpha);
          tmem_st32(tmem + lane_off + col_o + q4 * 32, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(bar(C::B_PFULL + sb));
    }
    // ------------------------------------------------------------ epilogue
    // With ROT3 the per-tile P V barrier can be two phases behind here (the
    // last S waited for implies only O += P_x(nt-3) V), so the epilogue waits
    // for the barrier committed once after the tile's last P V.  Without
    // ROT3 that S implies O += P_x(nt-2) V, and the per-tile barrier is at
    // most one phase behind.
    if (ok && nt > 0)
      ok = __all_sync(0xffffffffu,
                      C::ROT3 ? mbar_wait(bar(C::B_OFIN + x), 0, abort_flag, p.err,
                                          kErrTimeoutEpilogue)
                              : mbar_wait(bar(C::B_ODONE + x), (nt - 1) & 1, abort_flag, p.err,
                                          kErrTimeoutEpilogue));
    if (ok && nt > 0) {
      tc_fence_after();
      const float inv_l = p.o_scale / l;
      const bool live = qi < p.N;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.N + (live ? qi : 0)) * D;
#pragma unroll
      for (int q4 = 0; q4 < D / 32; ++q4) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + col_o + q4 * 32, r);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
          pk[t] = pack_bf16x2(__uint_as_float(r[2 * t]) * inv_l,
                              __uint_as_float(r[2 * t + 1]) * inv_l);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(orow + q4 * 32);
#pragma unroll
          for (int t = 0; t < 4; ++t)
            dst[t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
        }
      }
      if (live) p.lse[static_cast<size_t>(bh) * p.N + qi] = (m_used + log2f(l)) * kLn2;
    }
  }

  // Every warp reconverges first: in the TMA and MMA warps only one lane did
  // the work, and the CTA barrier below must count whole, converged warps.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool CAUSAL, bool FP8 = false>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         void* o, float* lse, const AttnShape& s, uint32_t* err,
                         cudaStream_t stream, float o_scale = 1.0f) {
  using C = FwdCfg<D, FP8>;
  auto kern = fa_fwd_kernel<D, CAUSAL, FP8>;
  cudaError_t e = set_smem_limit_once<fa_fwd_kernel<D, CAUSAL, FP8>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  FwdParams p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.N = s.N;
  p.Nk = s.keys();
  p.q_offset = s.q_offset;
  p.Hq = s.Hq;
  p.G = s.Hq / s.Hkv;
  p.n_qtiles = (s.N + C::BM - 1) / C::BM;
  p.n_qpairs = (p.n_qtiles + 1) / 2;
  p.n_ktiles = (p.Nk + C::BN - 1) / C::BN;
  p.scale_log2 = s.scale * kLog2e;
  p.o_scale = o_scale;
  p.err = err;
  p.n_heads = s.B * s.Hq;
  p.heads_per_group =
      static_cast<int>(heads_per_group(p.Nk, D, FP8 ? 1.0 : 2.0, p.G, p.n_heads));
  const long long grid = static_cast<long long>(s.B) * s.Hq * p.n_qpairs;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_dependent(kern, dim3(static_cast<unsigned>(grid)), dim3(C::THREADS), C::SMEM_BYTES,
                          stream, tq, tk, tv, p);
}

// Query rows per CTA: 128 (fa_fwd_tile1.cu) or 256 (two tiles here); 0 lets
// use_one_tile_per_cta decide per shape.
std::atomic<int> g_rows_per_cta{0};

// The per-shape choice between one and two query tiles per CTA.  Two tiles
// per CTA share each K/V tile between two softmax warpgroups and do more
// work per tile step; one tile per CTA makes twice as many, shorter CTAs,
// which wins while the two-tile grid would leave SMs idle or end on a short
// last wave.  Both kernels hold all 512 tensor-memory columns, so an SM runs
// one CTA at a time, and the choice is made by estimating each grid's finish
// time: the CTAs, in launch order, each start on the SM that frees first,
// and a CTA costs its per-CTA overhead plus its key-tile steps.  The costs,
// in units of one 128 x 128 key-tile step of the two-tile CTA, were fitted
// on GB300 to kernel times from CUDA-graph replay (152 SMs; d = 64, 96
// and 128, causal and not, B*H from 2 to 64, N from 1024 to 8192):
//   d = 64:  two-tile CTA steps,      one-tile CTA 1 + 1.35 x steps;
//   d = 96:  two-tile CTA 1 + steps,  one-tile CTA 2.5 + 1.05 x steps;
//   d = 128: two-tile CTA 1 + steps,  one-tile CTA 3 + 1.0 x steps.
// Past 16 two-tile waves the last wave no longer matters and the two-tile
// CTA's cheaper steps win.
std::mutex g_rows_mu;
std::map<std::array<long long, 8>, int> g_rows_cache;

double list_schedule_finish(int sms, long long n_heads, long long heads_per_group,
                            long long units, bool causal, const std::function<double(long long)>& cost) {
  std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
  for (int i = 0; i < sms; ++i) free_at.push(0.0);
  double finish = 0.0;
  for (long long g0 = 0; g0 < n_heads; g0 += heads_per_group) {
    const long long in_grp = std::min(heads_per_group, n_heads - g0);
    for (long long i = 0; i < units; ++i) {
      const double c = cost(causal ? units - 1 - i : i);
      for (long long h = 0; h < in_grp; ++h) {
        const double t = free_at.top() + c;
        free_at.pop();
        free_at.push(t);
        finish = std::max(finish, t);
      }
    }
  }
  return finish;
}

}  // namespace

int forward_rows_for(const AttnShape& s, int sms) {
  if (s.d == 256) return 128;
  if (s.d != 64 && s.d != 96 && s.d != 128) return 256;
  const long long n_qtiles = (static_cast<long long>(s.N) + 127) / 128;
  const long long n_ktiles = (static_cast<long long>(s.keys()) + 127) / 128;
  const long long n_pairs = (n_qtiles + 1) / 2;
  const long long n_heads = static_cast<long long>(s.B) * s.Hq;
  if (n_heads * n_pairs > 16LL * sms) return 256;
  const std::array<long long, 8> key{n_heads, s.Hq / s.Hkv, s.N, s.keys(), s.q_offset, s.d,
                                     s.causal ? 1 : 0, sms};
  {
    std::lock_guard<std::mutex> lk(g_rows_mu);
    const auto it = g_rows_cache.find(key);
    if (it != g_rows_cache.end()) return it->second;
  }
  // Launch-order grouping of heads, as both kernels' launches size it.
  const long long hpg = heads_per_group(s.keys(), s.d, 2.0, s.Hq / s.Hkv, n_heads);
  // Key tiles visited by query tile qt (the kernels' causal bound).
  auto tiles = [&](long long qt) -> double {
    if (qt >= n_qtiles) return 0.0;
    if (!s.causal) return static_cast<double>(n_ktiles);
    return static_cast<double>(std::min((s.q_offset + qt * 128 + 127) / 128 + 1, n_ktiles));
  };
  // Per-CTA overhead of the two-tile CTA; overhead and step cost of the
  // one-tile CTA (the fitted values listed above).
  const double o2 = s.d == 64 ? 0.0 : 1.0;
  const double o1 = s.d == 64 ? 1.0 : s.d == 96 ? 2.5 : 3.0;
  const double r1 = s.d == 64 ? 1.35 : s.d == 96 ? 1.05 : 1.0;
  const double pair = list_schedule_finish(sms, n_heads, hpg, n_pairs, s.causal != 0,
                                           [&](long long u) { return o2 + tiles(2 * u) + tiles(2 * u + 1); });
  const double one = list_schedule_finish(sms, n_heads, hpg, n_qtiles, s.causal != 0,
                                          [&](long long u) { return o1 + r1 * tiles(u); });
  const int rows = one < pair ? 128 : 256;
  std::lock_guard<std::mutex> lk(g_rows_mu);
  if (g_rows_cache.size() > 1024) g_rows_cache.clear();
  g_rows_cache.emplace(key, rows);
  return rows;
}

namespace {

bool use_one_tile_per_cta(const AttnShape& s) {
  const int forced = g_rows_per_cta.load(std::memory_order_relaxed);
  if (forced == 128) return true;
  if (forced == 256 || forced == 512) return false;
  static int sms = [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 148;
    return n;
  }();
  return forward_rows_for(s, sms) == 128;
}

}  // namespace

bool forward_uses_pair(const AttnShape& s) {
  return s.d == 128 && g_rows_per_cta.load(std::memory_order_relaxed) == 512;
}

void set_forward_rows_per_cta(int rows) { g_rows_per_cta.store(rows); }
int forward_rows_per_cta() { return g_rows_per_cta.load(); }

cudaError_t launch_forward(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           void* o, float* lse, const AttnShape& s, uint32_t* err,
                           cudaStream_t stream) {
  if (s.d == 256) return launch_forward_tile1(tq, tk, tv, o, lse, s, err, stream);
  if ((s.d == 64 || s.d == 96 || s.d == 128) && use_one_tile_per_cta(s))
    return launch_forward_tile1(tq, tk, tv, o, lse, s, err, stream);
  if (s.d == 64)
    return s.causal ? launch_fwd_t<64, true>(tq, tk, tv, o, lse, s, err, stream)
                    : launch_fwd_t<64, false>(tq, tk, tv, o, lse, s, err, stream);
  if (s.d == 96)
    return s.causal ? launch_fwd_t<96, true>(tq, tk, tv, o, lse, s, err, stream)
                    : launch_fwd_t<96, false>(tq, tk, tv, o, lse, s, err, stream);
  return s.causal ? launch_fwd_t<128, true>(tq, tk, tv, o, lse, s, err, stream)
                  : launch_fwd_t<128, false>(tq, tk, tv, o, lse, s, err, stream);
}

cudaError_t launch_forward_fp8(const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tvt, void* o, float* lse, const AttnShape& s,
                               float v_descale, uint32_t* err, cudaStream_t stream) {
  return s.causal ? launch_fwd_t<128, true, true>(tq, tk, tvt, o, lse, s, err, stream, v_descale)
                  : launch_fwd_t<128, false, true>(tq, tk, tvt, o, lse, s, err, stream, v_descale);
}

}  // namespace fa
