// Forward pass of exact attention on sm_103a for head dimension 128, with a
// pair of CTAs sharing their tensor-core products (tcgen05 cta_group::2).
//
// Same mathematics and the same per-CTA structure as fa_fwd.cu (two query
// tiles per CTA, one softmax warpgroup each, online softmax with the lazy
// rescale; "FlashAttention: l'attenzione che non spreca memoria", section
// "L'idea: lavorare a tessere, mai scrivere la matrice"; "L'attention
// fusionnee", section "Le softmax en ligne"), arranged so that two CTAs of a
// cluster run each product as one M = 256 MMA:
//
//  * The pair owns four consecutive query tiles of one (batch, query head):
//    CTA r (its rank in the cluster) holds tiles A_r = 4q + r and
//    B_r = 4q + 2 + r.  The "A" products cover tiles 4q and 4q + 1 (rows
//    0..127 of the MMA from CTA 0, 128..255 from CTA 1), the "B" products
//    4q + 2 and 4q + 3.  Under the causal mask each pair of tiles visits
//    the key tiles up to its later tile's last row; the earlier tile's rows
//    mask the excess.
//  * Each CTA loads half of every K tile (64 of its 128 keys, all of d) and
//    half of every V tile (all keys, 64 of the 128 columns of d): the B
//    operand of Q K^T is split by keys and that of P V by columns of d
//    between the two CTAs' shared memory.  Per SM that is half the K/V bytes
//    of fa_fwd.cu for half the products, which leaves room for four stages.
//  * One thread of CTA 0 issues every product; its commits arrive on the
//    barrier at the same offset in both CTAs.  A relay warp in each CTA
//    forwards "this CTA's half has landed" to CTA 0 (each CTA's copies
//    complete on its own barriers), and the softmax warps of both CTAs
//    arrive on CTA 0's P barriers.
//
// Warps (384 threads per CTA): 0-3 softmax of tile A, 4-7 softmax of tile B,
// 8 TMA producer, 9 MMA issuer (CTA 0) and tensor-memory owner, 10 relay,
// 11 idle.  Tensor memory per CTA: S_A [0,128), S_B [128,256) (P as packed
// bf16 over the first 64 columns), O_A [256,384), O_B [384,512).
//
// Every mbarrier wait is bounded (about a second); on expiry the CTA sets an
// error bit and skips its remaining work (the other CTA's waits then run out
// in turn); both CTAs meet at a cluster barrier before the tensor memory is
// released.

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

struct PairCfg {
  static constexpr int D = 128;
  static constexpr int BM = 128;                 // query rows per tile
  static constexpr int BN = 128;                 // keys per key tile
  static constexpr int QBLK = 128 * 128;         // 128 rows x 64 bf16 (128-byte swizzle)
  static constexpr int QTILE = 2 * QBLK;         // 128 x 128 query tile
  static constexpr int KHALF = 2 * 64 * 128;     // 64 keys x 128 d: two 8 KB blocks
  static constexpr int KBLK = 64 * 128;
  static constexpr int VHALF = 128 * 128;        // 128 keys x 64 d: one block
  static constexpr int NS = 4;                   // K/V ring stages
  static constexpr int OFF_Q = 0;                // tiles A and B
  static constexpr int OFF_K = OFF_Q + 2 * QTILE;
  static constexpr int OFF_V = OFF_K + NS * KHALF;
  static constexpr int OFF_BAR = OFF_V + NS * VHALF;
  // barrier slots (same layout in both CTAs)
  static constexpr int B_QFULL = 0;              // this CTA's Q tiles landed
  static constexpr int B_KFULL = 1;              // [NS] this CTA's K half landed
  static constexpr int B_VFULL = B_KFULL + NS;   // [NS]
  static constexpr int B_KEMPTY = B_VFULL + NS;  // [NS] K_j read by the pair's products
  static constexpr int B_VEMPTY = B_KEMPTY + NS; // [NS]
  static constexpr int B_QREADY = B_VEMPTY + NS; // CTA 0: both CTAs' Q landed (2 relays)
  static constexpr int B_KREADY = B_QREADY + 1;  // [NS] CTA 0: both K halves (2 relays)
  static constexpr int B_VREADY = B_KREADY + NS; // [NS]
  static constexpr int B_SFULL = B_VREADY + NS;  // [2] S of tile x in both CTAs
  static constexpr int B_PFULL = B_SFULL + 2;    // [2] CTA 0: P of tile x (8 warps, both CTAs)
  static constexpr int B_ODONE = B_PFULL + 2;    // [2] O += P V of tile x done
  static constexpr int B_DRAIN = B_ODONE + 2;    // abort path: products in flight
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = 256;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct PairParams {
  __nv_bfloat16* o;
  float* lse;
  int N, Nk, q_offset, Hq, G;
  int n_qtiles, n_quads, n_ktiles, n_heads, heads_per_group;
  float scale_log2;
  uint32_t* err;
};

template <bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const PairParams p) {
  using C = PairCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8 * i; };
  // The same barrier in CTA 0 of the pair (shared::cluster address).
  auto bar0 = [&](int i) -> uint32_t { return cluster_map(bar(i), 0); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const uint32_t rank = cluster_ctarank();
  // Launch order as in fa_fwd.cu, per pair of CTAs: groups of heads whose
  // K/V fit in L2, heaviest causal quads of tiles first.
  const int unit = static_cast<int>(blockIdx.x) >> 1;
  const int per_group = p.heads_per_group * p.n_quads;
  const int grp = unit / per_group;
  const int rem = unit - grp * per_group;
  const int in_grp = min(p.heads_per_group, p.n_heads - grp * p.heads_per_group);
  const int qi_ = rem / in_grp;
  const int bh = grp * p.heads_per_group + (rem - qi_ * in_grp);  // flattened (batch, query head)
  const int quad = CAUSAL ? (p.n_quads - 1 - qi_) : qi_;
  const int b = bh / p.Hq;
  const int hq = bh - b * p.Hq;
  const int kvz = b * (p.Hq / p.G) + hq / p.G;
  auto tiles_for = [&](int qt) -> int {
    if (qt >= p.n_qtiles) return 0;
    return CAUSAL ? min((p.q_offset + qt * C::BM + C::BM - 1) / C::BN + 1, p.n_ktiles)
                  : p.n_ktiles;
  };
  // Key tiles of the A products (tiles 4q, 4q + 1) and of the B products.
  const int nA = max(tiles_for(4 * quad), tiles_for(4 * quad + 1));
  const int nB = max(tiles_for(4 * quad + 2), tiles_for(4 * quad + 3));
  const int n_kv = max(nA, nB);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == C::B_QREADY || (i >= C::B_KREADY && i < C::B_SFULL)) cnt = 2;  // one relay per CTA
      if (i == C::B_PFULL || i == C::B_PFULL + 1) cnt = 8;  // softmax warps of both CTAs
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  // Both CTAs' barriers exist before either CTA arrives on the other's.
  cluster_sync_all();
  if (warp == 9) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dependency_wait();
  grid_launch_dependents();

  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t sK = sbase + C::OFF_K;
  const uint32_t sV = sbase + C::OFF_V;

  if (warp >= 8) {
    reg_decrease<56>();
    if (warp == 8) {
      // ---------------------------------------------------------- TMA producer
      if (elect_one()) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        const uint64_t keep = policy_evict_last();
        mbar_arrive_expect_tx(bar(C::B_QFULL), 2 * C::QTILE);
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int s = 0; s < 2; ++s)
            tma_load_3d(sQ + x * C::QTILE + s * C::QBLK, &tmQ, bar(C::B_QFULL), 64 * s,
                        (4 * quad + 2 * x + static_cast<int>(rank)) * C::BM, bh);
        int issued = 0;
        for (int j = 0; j < n_kv; ++j) {
          const int st = j % C::NS;
          const uint32_t ph = ((j / C::NS) - 1) & 1;
          if (j >= C::NS &&
              !mbar_wait(bar(C::B_KEMPTY + st), ph, abort_flag, p.err, kErrTimeoutLoad))
            break;
          // Keys 64 rank .. 64 rank + 63 of key tile j, all of d.
          mbar_arrive_expect_tx(bar(C::B_KFULL + st), C::KHALF);
#pragma unroll
          for (int s = 0; s < 2; ++s)
            tma_load_3d_hint(sK + st * C::KHALF + s * C::KBLK, &tmK, bar(C::B_KFULL + st), 64 * s,
                             j * C::BN + 64 * static_cast<int>(rank), kvz, keep);
          if (j >= C::NS &&
              !mbar_wait(bar(C::B_VEMPTY + st), ph, abort_flag, p.err, kErrTimeoutLoad))
            break;
          // All 128 keys of tile j, columns 64 rank .. 64 rank + 63 of d.
          mbar_arrive_expect_tx(bar(C::B_VFULL + st), C::VHALF);
          tma_load_3d_hint(sV + st * C::VHALF, &tmV, bar(C::B_VFULL + st),
                           64 * static_cast<int>(rank), j * C::BN, kvz, keep);
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
    } else if (warp == 10) {
      // ---------------------------------------------------------- relay
      // Tells CTA 0's issuer, in load order, that this CTA's Q, K and V
      // halves have landed.
      if (elect_one()) {
        bool ok = mbar_wait(bar(C::B_QFULL), 0, abort_flag, p.err, kErrTimeoutOther);
        if (ok) mbar_arrive_cluster(bar0(C::B_QREADY));
        for (int j = 0; ok && j < n_kv; ++j) {
          const int st = j % C::NS;
          const uint32_t ph = (j / C::NS) & 1;
          ok = mbar_wait(bar(C::B_KFULL + st), ph, abort_flag, p.err, kErrTimeoutOther);
          if (!ok) break;
          mbar_arrive_cluster(bar0(C::B_KREADY + st));
          ok = mbar_wait(bar(C::B_VFULL + st), ph, abort_flag, p.err, kErrTimeoutOther);
          if (!ok) break;
          mbar_arrive_cluster(bar0(C::B_VREADY + st));
        }
      }
    } else if (warp == 9 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer (CTA 0)
      // Order: S_A(0) S_B(0), then per key tile j: PV_A(j) S_A(j+1) PV_B(j)
      // S_B(j+1), as in fa_fwd.cu; each product covers both CTAs' tiles.
      if (elect_one()) {
        constexpr uint32_t ID_S = idesc_bf16_f32(256, 128, false, false);
        constexpr uint32_t ID_O = idesc_bf16_f32(256, 128, false, true);
        const uint64_t q_desc = smem_desc_sw128(sQ, 16, 1024);
        const uint64_t k_desc = smem_desc_sw128(sK, 16, 1024);       // 64 keys per CTA
        const uint64_t v_desc = smem_desc_sw128(sV, C::VHALF, 1024); // MN-major, 64 d per CTA
        const int nx[2] = {nA, nB};
        bool ok = mbar_wait_cluster(bar(C::B_QREADY), 0, abort_flag, p.err, kErrTimeoutMma);
        auto issue_s = [&](int x, int j) {
          const uint32_t d_tmem = tmem + x * 128;
          const uint64_t qd = desc_add(q_desc, x * C::QTILE);
          const uint64_t kd = desc_add(k_desc, (j % C::NS) * C::KHALF);
          mma_ss_pair<ID_S, 0>(d_tmem, qd, kd);
#pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            mma_ss_pair<ID_S, 1>(d_tmem, desc_add(qd, (kk >> 2) * C::QBLK + (kk & 3) * 32),
                                 desc_add(kd, (kk >> 2) * C::KBLK + (kk & 3) * 32));
          mma_commit_pair(bar(C::B_SFULL + x));
        };
        auto k_ready = [&](int j) -> bool {
          if (!mbar_wait_cluster(bar(C::B_KREADY + j % C::NS), (j / C::NS) & 1, abort_flag, p.err,
                                 kErrTimeoutMma))
            return false;
          tc_fence_after();
          return true;
        };
        if (ok && n_kv > 0) {
          ok = k_ready(0);
          if (ok) {
            if (nA > 0) issue_s(0, 0);
            if (nB > 0) issue_s(1, 0);
            mma_commit_pair(bar(C::B_KEMPTY + 0));
          }
        }
        for (int j = 0; ok && j < n_kv; ++j) {
          const int st = j % C::NS;
          if (!mbar_wait_cluster(bar(C::B_VREADY + st), (j / C::NS) & 1, abort_flag, p.err,
                                 kErrTimeoutMma))
            break;
          const bool next = j + 1 < n_kv;
          bool kn = false;
#pragma unroll 1
          for (int x = 0; x < 2; ++x) {
            if (j >= nx[x]) continue;
            if (!mbar_wait_cluster(bar(C::B_PFULL + x), j & 1, abort_flag, p.err,
                                   kErrTimeoutMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // O_x += P_x V_j: P packed over the first 64 columns of S_x, 16
            // keys (8 columns, 16 rows of V = 2 KB) per step.
            const uint64_t vd = desc_add(v_desc, st * C::VHALF);
            const uint32_t pa = tmem + x * 128;
            const uint32_t od = tmem + C::COL_O + x * 128;
            if (j == 0)
              mma_ts_pair<ID_O, 0>(od, pa, vd);
            else
              mma_ts_pair<ID_O, 1>(od, pa, vd);
#pragma unroll
            for (int kk = 1; kk < 8; ++kk)
              mma_ts_pair<ID_O, 1>(od, pa + kk * 8, desc_add(vd, kk * 2048));
            mma_commit_pair(bar(C::B_ODONE + x));
            if (next && j + 1 < nx[x]) {
              if (!kn) {
                if (!k_ready(j + 1)) {
                  ok = false;
                  break;
                }
                kn = true;
              }
              issue_s(x, j + 1);
            }
          }
          if (!ok) break;
          mma_commit_pair(bar(C::B_VEMPTY + st));
          if (kn) mma_commit_pair(bar(C::B_KEMPTY + (j + 1) % C::NS));
        }
        if (*abort_flag) {
          mma_commit_pair(bar(C::B_DRAIN));
          mbar_wait_timed(bar(C::B_DRAIN), 0);
        }
      }
    }
  } else {
    reg_increase<224>();
    // ------------------------------------------------------------ softmax (rows)
    const int x = warp >> 2;            // tile A or B of this CTA
    const int row = threadIdx.x & 127;  // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int qt = 4 * quad + 2 * x + static_cast<int>(rank);
    const int qi = qt * C::BM + row;
    const int nt = x == 0 ? nA : nB;    // the pair's product count for this tile
    const uint32_t col_s = x * 128;
    const uint32_t col_o = C::COL_O + x * 128;
    const uint32_t pfull0 = bar0(C::B_PFULL + x);
    const float c = p.scale_log2;
    float m_used = -INFINITY;
    float l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar(C::B_SFULL + x), j & 1, abort_flag,
                                                     p.err, kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
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
      const int qpos = p.q_offset + qi;
      const bool need_mask =
          (kbase + C::BN > p.Nk) || (CAUSAL && kbase + C::BN - 1 > p.q_offset + qt * C::BM);
      if (need_mask) {
#pragma unroll
        for (int t = 0; t < 128; ++t) {
          const int key = kbase + t;
          if (key >= p.Nk || (CAUSAL && key > qpos)) s[t] = -INFINITY;
        }
      }
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
      const uint64_t c2 = f2_pack(c, c);
      const uint64_t nm2 = f2_pack(-m_ref, -m_ref);
      uint64_t ps2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) ps2[u] = 0ull;
      {
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
        tmem_st32(tmem + lane_off + col_s, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(tmem + lane_off + col_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      }
      float sum, sum_hi;
      f2_unpack(f2_add(f2_add(ps2[0], ps2[1]), f2_add(ps2[2], ps2[3])), sum, sum_hi);
      sum += sum_hi;
      l = l * alpha + sum;
      // O holds P_0..P_{j-1} contributions; it must be final before it is
      // rescaled.  S_x(j) was issued after O += P_x(j-1) V by the same
      // thread, whose commit tracks every earlier product, so that product
      // has completed once S_x(j) has; the wait is kept for the rescale alone.
      // O += P_x(j) V waits for this tile's P (in both CTAs), so the barrier
      // is never two phases ahead of a waiter.
      const bool resc = j > 0 && __any_sync(0xffffffffu, upd);
      if (resc) {
        ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar(C::B_ODONE + x), (j - 1) & 1,
                                                       abort_flag, p.err, kErrTimeoutSoftmax));
        if (!ok) break;
      }
      if (resc) {
        tc_fence_after();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
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
      __syncwarp();
      if (lane_id() == 0) mbar_arrive_cluster(pfull0);  // on CTA 0's barrier
    }
    // ------------------------------------------------------------ epilogue
    if (ok && nt > 0)
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar(C::B_ODONE + x), (nt - 1) & 1,
                                                     abort_flag, p.err, kErrTimeoutEpilogue));
    if (ok && nt > 0) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const bool live = qi < p.N;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.N + (live ? qi : 0)) * C::D;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
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

  // Every warp reconverges; then both CTAs meet (no product reads either
  // CTA's memory any more, no arrival on CTA 0's barriers is in flight)
  // before the pair's tensor memory is released.
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

template <bool CAUSAL>
cudaError_t launch_pair_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          void* o, float* lse, const AttnShape& s, uint32_t* err,
                          cudaStream_t stream) {
  using C = PairCfg;
  auto kern = fa_fwd_pair_kernel<CAUSAL>;
  cudaError_t e = set_smem_limit_once<fa_fwd_pair_kernel<CAUSAL>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  PairParams p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.N = s.N;
  p.Nk = s.keys();
  p.q_offset = s.q_offset;
  p.Hq = s.Hq;
  p.G = s.Hq / s.Hkv;
  p.n_qtiles = (s.N + C::BM - 1) / C::BM;
  p.n_quads = (p.n_qtiles + 3) / 4;
  p.n_ktiles = (p.Nk + C::BN - 1) / C::BN;
  p.n_heads = s.B * s.Hq;
  p.heads_per_group = static_cast<int>(heads_per_group(p.Nk, C::D, 2.0, p.G, p.n_heads));
  p.scale_log2 = s.scale * kLog2e;
  p.err = err;
  const long long grid = 2LL * p.n_heads * p.n_quads;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

}  // namespace

// d = 128.  tk: K map with 64 x 64 boxes (half a key tile); tv: V map with
// 64 x 128 boxes; tq: the usual 64 x 128 query boxes.
cudaError_t launch_forward_pair(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, void* o, float* lse, const AttnShape& s,
                                uint32_t* err, cudaStream_t stream) {
  if (s.d != 128) return cudaErrorInvalidValue;
  return s.causal ? launch_pair_t<true>(tq, tk, tv, o, lse, s, err, stream)
                  : launch_pair_t<false>(tq, tk, tv, o, lse, s, err, stream);
}

}  // namespace fa
