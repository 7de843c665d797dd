// Forward pass of exact attention on sm_103a with one query tile per CTA.
//
// Same mathematics as fa_fwd.cu ("FlashAttention: l'attenzione che non spreca
// memoria", section "L'idea: lavorare a tessere, mai scrivere la matrice";
// online softmax as in "L'attention fusionnee", section "Le softmax en
// ligne") with a query block of B_r = 128 rows per CTA instead of fa_fwd.cu's
// two tiles (B_r = 256).  It is the only forward for d = 256 (a 128 x 256
// bf16 query tile is 64 KB and its fp32 O takes 256 of the 512 TMEM columns,
// so keys come in tiles of 64 there), and the alternative tile size for
// d = 64, 96 and 128 (keys in tiles of 128): twice as many CTAs, which covers
// the SMs better when there are few query tiles.
//
// Pipeline: the S tile of key tile j is computed into tensor-memory buffer
// j mod 3, so the tensor core computes S_{j+1} and S_{j+2} (and O += P_j V_j)
// while the softmax warpgroup turns S_j into P_j.  The buffer that
// O += P_j V_j reads is next overwritten by S_{j+3}, issued after the
// following O += P V product.
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t; online softmax with the
//              lazy rescale of fa_fwd.cu (the reference maximum moves only
//              when the running maximum has grown by more than
//              kRescaleThreshold in log2 units), epilogue.
//   warp 4     TMA producer: the query tile once, then K_j and V_j into a
//              two-stage ring.
//   warp 5     MMA issuer and TMEM owner: S_0, S_1, then per key tile j:
//              O += P_j V_j, S_{j+2} = Q K_{j+2}^T into buffer (j+2) mod 3.
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   columns BN*b .. BN*b + BN - 1   S buffer b = 0, 1, 2 (P as packed bf16
//                                   over its first BN/2 columns)
//   columns 512 - DP .. 512 - DP + D - 1   O accumulator (fp32; DP = D
//                                   rounded up to a multiple of 64)
//
// Every mbarrier wait is bounded (about a second); on expiry the kernel sets
// an error bit, every role skips its remaining work and the CTA exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

template <int D_>
struct Cfg1 {
  static constexpr int D = D_;                   // 64, 96, 128 or 256
  // Tiles are stored DP = D rounded up to whole 128-byte swizzle atoms wide;
  // at D = 96 the copies fill columns 96..127 with zeros (outside the
  // tensor), Q K^T runs its 16-column k-steps over the first 96 and
  // O += P V has N = 96.
  static constexpr int DP = (D + 63) / 64 * 64;
  static constexpr int BM = 128;                 // query rows per tile (MMA M)
  static constexpr int BN = D == 256 ? 64 : 128; // keys per tile (MMA N of Q K^T)
  static constexpr int SUB = DP / 64;            // 128-byte column blocks per row
  static constexpr int Q_BLOCK = BM * 128;       // one 128-row x 64-col block
  static constexpr int KV_BLOCK = BN * 128;      // one BN-row x 64-col block
  static constexpr int Q_TILE = SUB * Q_BLOCK;
  static constexpr int KV_TILE = SUB * KV_BLOCK;
  static constexpr int NS = D == 64 ? 4 : 2;     // K/V ring stages
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_TILE;
  static constexpr int OFF_V = OFF_K + NS * KV_TILE;
  static constexpr int OFF_BAR = OFF_V + NS * KV_TILE;
  // barrier slots
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;
  static constexpr int B_KEMPTY = B_KFULL + NS;
  static constexpr int B_VFULL = B_KEMPTY + NS;
  static constexpr int B_VEMPTY = B_VFULL + NS;
  static constexpr int NB = 3;                   // S/P buffers in tensor memory
  static constexpr int B_SFULL = B_VEMPTY + NS;  // [NB] S_j in buffer j % NB
  static constexpr int B_PFULL = B_SFULL + NB;   // [NB] P_j in buffer j % NB (4 warp arrivals)
  static constexpr int B_ODONE = B_PFULL + NB;   // O += P_j V_j completed
  static constexpr int B_FINAL = B_ODONE + 1;    // every product completed (once)
  static constexpr int B_DRAIN = B_FINAL + 1;    // abort path: MMAs in flight
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;  // tmem slot, abort word
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static constexpr int THREADS = 192;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = 512 - DP;  // above the NB S buffers
  static_assert(NB * BN <= 512 - DP, "tensor memory");
};

struct Fwd1Params {
  __nv_bfloat16* o;
  float* lse;
  int N;         // query rows
  int Nk;        // key/value rows
  int q_offset;  // absolute position of query row 0
  int Hq;
  int G;          // query heads per key/value head
  int n_qtiles;
  int n_ktiles;
  int n_heads;          // B * Hq
  int heads_per_group;  // launch-order grouping, a multiple of G
  float scale_log2;     // scale * log2(e)
  uint32_t* err;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(192, 1)
    fa_fwd1_kernel(const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const Fwd1Params p) {
  using C = Cfg1<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  // Launch order as in fa_fwd.cu: groups of heads whose K/V fit in L2, the
  // heaviest causal query tiles of the group first.
  const int per_group = p.heads_per_group * p.n_qtiles;
  const int grp = static_cast<int>(blockIdx.x) / per_group;
  const int rem = static_cast<int>(blockIdx.x) - grp * per_group;
  const int in_grp = min(p.heads_per_group, p.n_heads - grp * p.heads_per_group);
  const int qi_ = rem / in_grp;
  const int bh = grp * p.heads_per_group + (rem - qi_ * in_grp);  // flattened (batch, query head)
  const int qt = CAUSAL ? (p.n_qtiles - 1 - qi_) : qi_;
  const int b = bh / p.Hq;
  const int hq = bh - b * p.Hq;
  const int kvz = b * (p.Hq / p.G) + hq / p.G;  // flattened (batch, kv head)
  // Key tiles up to the one holding the last row's position (causal).
  const int n_kv = CAUSAL ? min((p.q_offset + qt * C::BM + C::BM - 1) / C::BN + 1, p.n_ktiles)
                          : p.n_ktiles;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_QFULL), 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 1);
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int x = 0; x < C::NB; ++x) mbar_init(bar(C::B_SFULL + x), 1);
    // One P barrier per buffer: the softmax may finish P_j and P_{j+1} before
    // the issuer waits for P_j, which one barrier could not tell apart by parity.
    for (int x = 0; x < C::NB; ++x) mbar_init(bar(C::B_PFULL + x), 4);  // one per softmax warp
    mbar_init(bar(C::B_ODONE), 1);
    mbar_init(bar(C::B_FINAL), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
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

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t keep = policy_evict_last();  // K/V are re-read by the other query tiles
      mbar_arrive_expect_tx(bar(C::B_QFULL), C::Q_TILE);
#pragma unroll
      for (int s = 0; s < C::SUB; ++s)
        tma_load_3d(sQ + s * C::Q_BLOCK, &tmQ, bar(C::B_QFULL), 64 * s, qt * C::BM, bh);
      int issued = 0;  // K/V tiles whose loads were issued
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % C::NS;
        const uint32_t ph = ((j / C::NS) - 1) & 1;
        if (j >= C::NS &&
            !mbar_wait(bar(C::B_KEMPTY + st), ph, abort_flag, p.err, kErrTimeoutLoad))
          break;
        mbar_arrive_expect_tx(bar(C::B_KFULL + st), C::KV_TILE);
#pragma unroll
        for (int s = 0; s < C::SUB; ++s)
          tma_load_3d_hint(sK + st * C::KV_TILE + s * C::KV_BLOCK, &tmK, bar(C::B_KFULL + st),
                           64 * s, j * C::BN, kvz, keep);
        if (j >= C::NS &&
            !mbar_wait(bar(C::B_VEMPTY + st), ph, abort_flag, p.err, kErrTimeoutLoad))
          break;
        mbar_arrive_expect_tx(bar(C::B_VFULL + st), C::KV_TILE);
#pragma unroll
        for (int s = 0; s < C::SUB; ++s)
          tma_load_3d_hint(sV + st * C::KV_TILE + s * C::KV_BLOCK, &tmV, bar(C::B_VFULL + st),
                           64 * s, j * C::BN, kvz, keep);
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
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t ID_S = idesc_bf16_f32(128, C::BN, false, false);
      constexpr uint32_t ID_O = idesc_bf16_f32(128, C::D, false, true);
      const uint64_t q_desc = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t k_desc = smem_desc_sw128(sK, 16, 1024);
      const uint64_t v_desc = smem_desc_sw128(sV, C::KV_BLOCK, 1024);  // MN-major, N = D
      bool ok = mbar_wait(bar(C::B_QFULL), 0, abort_flag, p.err, kErrTimeoutMma);
      // S_j = Q K_j^T into buffer j % NB (16 steps of 16 columns of d); K_j is
      // released when the product is done.
      auto issue_s = [&](int j) -> bool {
        const int st = j % C::NS;
        if (!mbar_wait(bar(C::B_KFULL + st), (j / C::NS) & 1, abort_flag, p.err, kErrTimeoutMma))
          return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (j % C::NB) * C::BN;
        const uint64_t kd = desc_add(k_desc, st * C::KV_TILE);
        mma_ss_k<ID_S, 0>(d_tmem, q_desc, kd);
#pragma unroll
        for (int kk = 1; kk < C::D / 16; ++kk)
          mma_ss_k<ID_S, 1>(d_tmem, desc_add(q_desc, (kk >> 2) * C::Q_BLOCK + (kk & 3) * 32),
                            desc_add(kd, (kk >> 2) * C::KV_BLOCK + (kk & 3) * 32));
        mma_commit(bar(C::B_SFULL + j % C::NB));
        mma_commit(bar(C::B_KEMPTY + st));
        return true;
      };
      for (int j = 0; ok && j < min(n_kv, 2); ++j) ok = issue_s(j);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % C::NS;
        const int bf = j % C::NB;
        if (!mbar_wait(bar(C::B_VFULL + st), (j / C::NS) & 1, abort_flag, p.err, kErrTimeoutMma))
          break;
        if (!mbar_wait(bar(C::B_PFULL + bf), (j / C::NB) & 1, abort_flag, p.err, kErrTimeoutMma))
          break;
        tc_fence_after();
        // O += P_j V_j: P packed in the first 32 columns of buffer bf, 16 keys
        // (8 columns, 16 rows of V = 2 KB) per step.
        const uint64_t vd = desc_add(v_desc, st * C::KV_TILE);
        const uint32_t pa = tmem + bf * C::BN;
        if (j == 0)
          mma_ts_k<ID_O, 0>(tmem + C::COL_O, pa, vd);
        else
          mma_ts_k<ID_O, 1>(tmem + C::COL_O, pa, vd);
#pragma unroll
        for (int kk = 1; kk < C::BN / 16; ++kk)
          mma_ts_k<ID_O, 1>(tmem + C::COL_O, pa + kk * 8, desc_add(vd, kk * 2048));
        mma_commit(bar(C::B_ODONE));
        mma_commit(bar(C::B_VEMPTY + st));
        // Once, after the last product: the softmax does not wait for every
        // O += P V, so at its epilogue the per-tile barrier may be two phases
        // behind, which parity cannot tell from "done".
        if (j == n_kv - 1) mma_commit(bar(C::B_FINAL));
        // S_{j+2} into buffer (j+2) % NB, whose P_{j-1} the previous O += P V
        // read.
        if (j + 2 < n_kv && !issue_s(j + 2)) break;
      }
      if (*abort_flag) {
        // Let the MMAs already issued finish before tensor memory is released.
        mma_commit(bar(C::B_DRAIN));
        mbar_wait_timed(bar(C::B_DRAIN), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax (rows)
    const int row = threadIdx.x;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int qi = qt * C::BM + row;
    const int qpos = p.q_offset + qi;  // absolute position of this row
    const float c = p.scale_log2;
    float m_used = -INFINITY;  // reference maximum, log2 domain
    float l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int bf = j % C::NB;
      const uint32_t col_s = bf * C::BN;
      // Waits are made warp-uniform: the TMEM loads and stores below are
      // warp-collective, so either every lane goes on or every lane stops.
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SFULL + bf), (j / C::NB) & 1, abort_flag,
                                             p.err, kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      // The row's scores: all loads in flight, one wait.
      float s[C::BN];
      {
        uint32_t r[C::BN];
#pragma unroll
        for (int q4 = 0; q4 < C::BN / 32; ++q4)
          tmem_ld32(tmem + lane_off + col_s + q4 * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(&r[q4 * 32]));
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < C::BN; ++t) s[t] = __uint_as_float(r[t]);
      }
      const int kbase = j * C::BN;
      const bool need_mask =
          (kbase + C::BN > p.Nk) || (CAUSAL && kbase + C::BN - 1 > p.q_offset + qt * C::BM);
      if (need_mask) {
#pragma unroll
        for (int t = 0; t < C::BN; ++t) {
          const int key = kbase + t;
          if (key >= p.Nk || (CAUSAL && key > qpos)) s[t] = -INFINITY;
        }
      }
      // Row max over 8 independent partial maxima, two new values per
      // three-input max.
      float pm[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) pm[u] = fmaxf(s[u], s[u + 8]);
#pragma unroll
      for (int t = 16; t < C::BN; t += 16)
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
      {
        uint32_t pk[C::BN / 2];
#pragma unroll
        for (int t = 0; t < C::BN / 2; ++t) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(s[2 * t], s[2 * t + 1]), c2, nm2), x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          ps2[t & 3] = f2_add(ps2[t & 3], f2_pack(p0, p1));
          pk[t] = pack_bf16x2(p0, p1);
        }
        // P over the S columns just read.
#pragma unroll
        for (int q4 = 0; q4 < C::BN / 64; ++q4)
          tmem_st32(tmem + lane_off + col_s + q4 * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(&pk[q4 * 32]));
      }
      float sum, sum_hi;
      f2_unpack(f2_add(f2_add(ps2[0], ps2[1]), f2_add(ps2[2], ps2[3])), sum, sum_hi);
      sum += sum_hi;
      l = l * alpha + sum;
      if (j > 0 && __any_sync(0xffffffffu, upd)) {
        // O holds P_0..P_{j-1} contributions; it must be final before rescaling
        // (O += P_j V_j is not issued before this warpgroup's P_j arrives).
        // S_j being ready implies O += P_{j-2} V_{j-2} is done (it was issued
        // before S_j), so the per-tile barrier is at most one phase behind.
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_ODONE), (j - 1) & 1, abort_flag, p.err,
                                               kErrTimeoutSoftmax));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int q4 = 0; q4 < C::D / 32; ++q4) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + C::COL_O + q4 * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 32; ++t) r[t] = __float_as_uint(__uint_as_float(r[t]) * alpha);
          tmem_st32(tmem + lane_off + C::COL_O + q4 * 32, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(bar(C::B_PFULL + bf));
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n_kv > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_FINAL), 0, abort_flag, p.err,
                                             kErrTimeoutEpilogue));
    if (ok && n_kv > 0) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const bool live = qi < p.N;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.N + (live ? qi : 0)) * C::D;
#pragma unroll 1
      for (int q4 = 0; q4 < C::D / 32; ++q4) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::COL_O + q4 * 32, r);
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
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* o,
                     float* lse, const AttnShape& s, uint32_t* err, cudaStream_t stream) {
  using C = Cfg1<D>;
  auto kern = fa_fwd1_kernel<D, CAUSAL>;
  cudaError_t e = set_smem_limit_once<fa_fwd1_kernel<D, CAUSAL>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  Fwd1Params p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.N = s.N;
  p.Nk = s.keys();
  p.q_offset = s.q_offset;
  p.Hq = s.Hq;
  p.G = s.Hq / s.Hkv;
  p.n_qtiles = (s.N + C::BM - 1) / C::BM;
  p.n_ktiles = (p.Nk + C::BN - 1) / C::BN;
  p.n_heads = s.B * s.Hq;
  p.scale_log2 = s.scale * kLog2e;
  p.err = err;
  p.heads_per_group = static_cast<int>(heads_per_group(p.Nk, C::D, 2.0, p.G, p.n_heads));
  const long long grid = static_cast<long long>(p.n_heads) * p.n_qtiles;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_dependent(kern, dim3(static_cast<unsigned>(grid)), dim3(C::THREADS), C::SMEM_BYTES,
                          stream, tq, tk, tv, p);
}

}  // namespace

// d in {64, 96, 128, 256}.  K and V maps have boxes of one key tile (64 rows
// for d = 256, else 128) x 64 columns; the query map boxes of 128 x 64.
cudaError_t launch_forward_tile1(const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, void* o, float* lse, const AttnShape& s,
                                 uint32_t* err, cudaStream_t stream) {
  if (s.d == 256)
    return s.causal ? launch_t<256, true>(tq, tk, tv, o, lse, s, err, stream)
                    : launch_t<256, false>(tq, tk, tv, o, lse, s, err, stream);
  if (s.d == 128)
    return s.causal ? launch_t<128, true>(tq, tk, tv, o, lse, s, err, stream)
                    : launch_t<128, false>(tq, tk, tv, o, lse, s, err, stream);
  if (s.d == 96)
    return s.causal ? launch_t<96, true>(tq, tk, tv, o, lse, s, err, stream)
                    : launch_t<96, false>(tq, tk, tv, o, lse, s, err, stream);
  if (s.d == 64)
    return s.causal ? launch_t<64, true>(tq, tk, tv, o, lse, s, err, stream)
                    : launch_t<64, false>(tq, tk, tv, o, lse, s, err, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
