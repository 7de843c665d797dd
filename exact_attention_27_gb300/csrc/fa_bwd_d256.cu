// dK/dV kernel of the backward pass for head dimension 256 on sm_103a.
//
// Mathematics of "L'attention fusionnee", section "La passe arriere :
// recalculer plutot que garder": P rebuilt from the saved L, dV = P^T dO,
// dS = P o (dP - D), dK = dS^T Q scale (dQ is computed by the dQ kernel of
// fa_bwd_dq.cu, which walks the key tiles of each query tile in the forward
// pass's order, so the whole d = 256 backward is free of atomics).
//
// Why this shape.  At d = 256 the fp32 dK and dV of a 128-key tile, with
// keys on the tensor-memory lanes as the d <= 128 kernels hold them, would
// fill all 512 TMEM columns before S or dP had any.  Here the accumulators
// are kept transposed instead: dV^T = dO^T P and dK^T = Q^T dS, with the head
// dimension on the lanes (two halves of 128) and the keys of a 64-key tile on
// the columns, 2 x 64 columns each.  One CTA owns 64 keys of one (batch,
// K/V head) and walks the 128-row query tiles of every query head of the
// group that see them:
//
//   dP   = dO_i V_j^T      tcgen05.mma  M 128 queries, N 64 keys, K 256
//   S    = Q_i K_j^T       tcgen05.mma  (issued after dP: Q_i is the last
//                          operand freed by the step before)
//   P    = exp2(S scale log2e - L log2e)          query-row threads
//   dV^T += dO_i^T P       two MMAs (d halves), A = dO_i read MN-major,
//                          B = P (bf16, written to shared memory as
//                          [query][key], read MN-major)
//   dS   = P o (dP - D)                           query-row threads
//   dK^T += Q_i^T dS       two MMAs, as dV^T
//
// Each query row belongs to one thread per half of the key tile (two warps
// per 32 rows), so L and D are per-thread scalars and no row reduction is
// needed.  dV^T is computed while the threads turn dP into dS.  At the end
// dK (times scale) and dV are written transposed back to [key][d].
//
// Warps: 0-7 query rows (warp w: rows 32 (w % 4).., keys 32 (w / 4)..),
// 8 TMA producer, 9 MMA issuer and tensor-memory owner.  320 threads.
// Tensor memory: dV^T [0,128) (half h at 64 h), dK^T [128,256), S [256,320),
// dP [320,384).
// Shared memory: K, V (64 x 256 bf16, 32 KB each), Q, dO (128 x 256 bf16,
// 64 KB each), P, dS (128 x 64 bf16, 16 KB each) = 224 KB.  One stage of
// each: at 128 rows of 512 bytes, a second Q/dO stage does not fit.  So Q
// and dO are split into two halves of d (128 columns) with a barrier each:
// the MMA issuer starts a product on half 0 while half 1 is still landing,
// and the producer reloads a half as soon as the dV^T / dK^T products that
// read it are done, rather than after both halves are.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct Kv256Cfg {
  static constexpr int D = 256;
  static constexpr int BK = 64;                    // keys per CTA
  static constexpr int BQ = 128;                   // queries per step
  static constexpr int KSUB = 64 * 128;            // 64 rows x 64 bf16
  static constexpr int QSUB = 128 * 128;           // 128 rows x 64 bf16
  static constexpr int KTILE = 4 * KSUB;
  static constexpr int QTILE = 4 * QSUB;
  static constexpr int PBYTES = 128 * 128;         // 128 query rows x 64 keys bf16
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KTILE;
  static constexpr int OFF_Q = OFF_V + KTILE;
  static constexpr int OFF_DO = OFF_Q + QTILE;
  static constexpr int OFF_P = OFF_DO + QTILE;
  static constexpr int OFF_DS = OFF_P + PBYTES;
  static constexpr int OFF_BAR = OFF_DS + PBYTES;
  // Q and dO are handled as two halves of d (128 columns, 32 KB each), so
  // that each half is reloaded as soon as the products reading it are done.
  static constexpr int B_KV = 0;
  static constexpr int B_QFULL = 1;      // [2] Q half landed
  static constexpr int B_DOFULL = 3;     // [2]
  static constexpr int B_QEMPTY = 5;     // [2] dK^T[h] of the step done: Q half h free
  static constexpr int B_DOEMPTY = 7;    // [2] dV^T[h] of the step done: dO half h free
  static constexpr int B_S = 9;          // S in tensor memory
  static constexpr int B_DP = 10;        // dP in tensor memory
  static constexpr int B_P = 11;         // P in shared memory, S read (8 warp arrivals)
  static constexpr int B_DS = 12;        // dS in shared memory, dP read (8 warp arrivals)
  static constexpr int B_PFREE = 13;     // dV^T done: P buffer free
  static constexpr int B_DSFREE = 14;    // dK^T done: dS buffer free
  static constexpr int B_FINAL = 15;     // every product issued has completed (once)
  static constexpr int B_DRAIN = 16;
  static constexpr int NBAR = 17;
  static constexpr int QHALF = 2 * QSUB;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 320;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_DV = 0, COL_DK = 128, COL_S = 256, COL_DP = 320;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct Kv256Params {
  const float* lse;
  const float* Dvec;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int N, Hq, Hkv, G, n_qtiles, n_ktiles;
  float scale;
  float scale_log2;
  uint32_t* err;
};

__device__ __forceinline__ uint32_t sw128(int r, int ch) {
  return static_cast<uint32_t>(r * 128 + ((ch ^ (r & 7)) << 4));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

template <bool CAUSAL>
__global__ void __launch_bounds__(320, 1)
    fa_bwd256_kv_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmdO, const Kv256Params p) {
  using C = Kv256Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  // Heaviest key tiles (most query tiles under the causal mask) first.
  const int n_kv_units = static_cast<int>(gridDim.x) / p.n_ktiles;
  const int jt = static_cast<int>(blockIdx.x) / n_kv_units;
  const int kvz = static_cast<int>(blockIdx.x) - jt * n_kv_units;  // flattened (batch, kv head)
  const int b = kvz / p.Hkv;
  const int hkv = kvz - b * p.Hkv;
  // Query tile i sees key tile jt (keys 64 jt ..) iff its last row 128 i + 127 >= 64 jt.
  const int i0 = CAUSAL ? (jt * C::BK) / C::BQ : 0;
  const int per_head = p.n_qtiles - i0;
  const int n_steps = p.G * per_head;

  const uint32_t sK = sbase + C::OFF_K;
  const uint32_t sV = sbase + C::OFF_V;
  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t sdO = sbase + C::OFF_DO;
  const uint32_t sP = sbase + C::OFF_P;
  const uint32_t sDS = sbase + C::OFF_DS;

  // step -> (flattened query head, query tile)
  auto step_coords = [&](int s, int& bhq, int& it) {
    const int g = s / per_head;
    it = i0 + (s - g * per_head);
    bhq = b * p.Hq + hkv * p.G + g;
  };

  if (warp == 8 && elect_one()) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    for (int i = 0; i < C::NBAR; ++i) mbar_init(bar(i), (i == C::B_P || i == C::B_DS) ? 8 : 1);
    *abort_flag = 0;
    fence_barrier_init();
    // K, V and step 0's dO and Q are inputs of the backward, which this grid
    // may read before it waits for the grid before it.
    mbar_arrive_expect_tx(bar(C::B_KV), 2 * C::KTILE);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      tma_load_3d(sK + c * C::KSUB, &tmK, bar(C::B_KV), 64 * c, jt * C::BK, kvz);
      tma_load_3d(sV + c * C::KSUB, &tmV, bar(C::B_KV), 64 * c, jt * C::BK, kvz);
    }
    if (n_steps > 0) {
      int bhq, it;
      step_coords(0, bhq, it);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mbar_arrive_expect_tx(bar(C::B_DOFULL + h), C::QHALF);
        for (int c = 2 * h; c < 2 * h + 2; ++c)
          tma_load_3d(sdO + c * C::QSUB, &tmdO, bar(C::B_DOFULL + h), 64 * c, it * C::BQ, bhq);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mbar_arrive_expect_tx(bar(C::B_QFULL + h), C::QHALF);
        for (int c = 2 * h; c < 2 * h + 2; ++c)
          tma_load_3d(sQ + c * C::QSUB, &tmQ, bar(C::B_QFULL + h), 64 * c, it * C::BQ, bhq);
      }
    }
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      // dO of step s once dV^T of step s - 1 has read its buffer, then Q once
      // dK^T has; step 0 was issued before the CTA barrier.
      int do_half[2], q_half[2];  // steps whose half h was issued
      do_half[0] = do_half[1] = q_half[0] = q_half[1] = n_steps > 0 ? 1 : 0;
      for (int s = 1; s < n_steps; ++s) {
        int bhq, it;
        step_coords(s, bhq, it);
        // Halves in the order the products free them: dO[0], dO[1] (dV^T),
        // then Q[0], Q[1] (dK^T).
        bool go = true;
#pragma unroll 1
        for (int h = 0; h < 2 && go; ++h) {
          if (!mbar_wait(bar(C::B_DOEMPTY + h), (s - 1) & 1, abort_flag, p.err, kErrTimeoutLoad)) {
            go = false;
            break;
          }
          mbar_arrive_expect_tx(bar(C::B_DOFULL + h), C::QHALF);
          for (int c = 2 * h; c < 2 * h + 2; ++c)
            tma_load_3d(sdO + c * C::QSUB, &tmdO, bar(C::B_DOFULL + h), 64 * c, it * C::BQ, bhq);
          do_half[h] = s + 1;
        }
#pragma unroll 1
        for (int h = 0; h < 2 && go; ++h) {
          if (!mbar_wait(bar(C::B_QEMPTY + h), (s - 1) & 1, abort_flag, p.err, kErrTimeoutLoad)) {
            go = false;
            break;
          }
          mbar_arrive_expect_tx(bar(C::B_QFULL + h), C::QHALF);
          for (int c = 2 * h; c < 2 * h + 2; ++c)
            tma_load_3d(sQ + c * C::QSUB, &tmQ, bar(C::B_QFULL + h), 64 * c, it * C::BQ, bhq);
          q_half[h] = s + 1;
        }
        if (!go) break;
      }
      if (*abort_flag) {
        mbar_wait_timed(bar(C::B_KV), 0);
        for (int h = 0; h < 2; ++h) {
          if (do_half[h] > 0) mbar_wait_timed(bar(C::B_DOFULL + h), (do_half[h] - 1) & 1);
          if (q_half[h] > 0) mbar_wait_timed(bar(C::B_QFULL + h), (q_half[h] - 1) & 1);
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t ID_SP = idesc_bf16_f32(128, 64, false, false);  // S, dP
      constexpr uint32_t ID_T = idesc_bf16_f32(128, 64, true, true);     // dV^T, dK^T
      const uint64_t q_k = smem_desc_sw128(sQ, 16, 1024);      // Q, K-major A
      const uint64_t do_k = smem_desc_sw128(sdO, 16, 1024);
      const uint64_t k_k = smem_desc_sw128(sK, 16, 1024);      // K, K-major B
      const uint64_t v_k = smem_desc_sw128(sV, 16, 1024);
      const uint64_t q_mn = smem_desc_sw128(sQ, C::QSUB, 1024);   // Q^T, MN-major A
      const uint64_t do_mn = smem_desc_sw128(sdO, C::QSUB, 1024);
      const uint64_t p_mn = smem_desc_sw128(sP, C::PBYTES, 1024);  // P, MN-major B (N = 64)
      const uint64_t ds_mn = smem_desc_sw128(sDS, C::PBYTES, 1024);
      bool ok = mbar_wait(bar(C::B_KV), 0, abort_flag, p.err, kErrTimeoutMma);
      for (int s = 0; ok && s < n_steps; ++s) {
        const uint32_t ph = s & 1;
        // dP = dO V^T (the dP columns were read by the threads of step s - 1
        // before they arrived on B_DS, which the previous iteration waited for).
        if (!mbar_wait(bar(C::B_DOFULL), ph, abort_flag, p.err, kErrTimeoutMma)) break;
        tc_fence_after();
        mma_ss_k<ID_SP, 0>(tmem + C::COL_DP, do_k, v_k);
#pragma unroll
        for (int kk = 1; kk < 8; ++kk)
          mma_ss_k<ID_SP, 1>(tmem + C::COL_DP,
                             desc_add(do_k, (kk >> 2) * C::QSUB + (kk & 3) * 32),
                             desc_add(v_k, (kk >> 2) * C::KSUB + (kk & 3) * 32));
        if (!mbar_wait(bar(C::B_DOFULL + 1), ph, abort_flag, p.err, kErrTimeoutMma)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 8; kk < 16; ++kk)
          mma_ss_k<ID_SP, 1>(tmem + C::COL_DP,
                             desc_add(do_k, (kk >> 2) * C::QSUB + (kk & 3) * 32),
                             desc_add(v_k, (kk >> 2) * C::KSUB + (kk & 3) * 32));
        mma_commit(bar(C::B_DP));
        // S = Q K^T
        if (!mbar_wait(bar(C::B_QFULL), ph, abort_flag, p.err, kErrTimeoutMma)) break;
        tc_fence_after();
        mma_ss_k<ID_SP, 0>(tmem + C::COL_S, q_k, k_k);
#pragma unroll
        for (int kk = 1; kk < 8; ++kk)
          mma_ss_k<ID_SP, 1>(tmem + C::COL_S,
                             desc_add(q_k, (kk >> 2) * C::QSUB + (kk & 3) * 32),
                             desc_add(k_k, (kk >> 2) * C::KSUB + (kk & 3) * 32));
        if (!mbar_wait(bar(C::B_QFULL + 1), ph, abort_flag, p.err, kErrTimeoutMma)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 8; kk < 16; ++kk)
          mma_ss_k<ID_SP, 1>(tmem + C::COL_S,
                             desc_add(q_k, (kk >> 2) * C::QSUB + (kk & 3) * 32),
                             desc_add(k_k, (kk >> 2) * C::KSUB + (kk & 3) * 32));
        mma_commit(bar(C::B_S));
        // dV^T[h] += dO^T[h] P: 128 queries in 8 steps of 16 rows (2 KB).
        if (!mbar_wait(bar(C::B_P), ph, abort_flag, p.err, kErrTimeoutMma)) break;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint64_t a = desc_add(do_mn, 2 * h * C::QSUB);
          const uint32_t dst = tmem + C::COL_DV + 64 * h;
          if (s == 0)
            mma_ss_k<ID_T, 0>(dst, a, p_mn);
          else
            mma_ss_k<ID_T, 1>(dst, a, p_mn);
#pragma unroll
          for (int kq = 1; kq < 8; ++kq)
            mma_ss_k<ID_T, 1>(dst, desc_add(a, kq * 2048), desc_add(p_mn, kq * 2048));
          mma_commit(bar(C::B_DOEMPTY + h));  // dO half h is no longer read
        }
        mma_commit(bar(C::B_PFREE));
        // dK^T[h] += Q^T[h] dS
        if (!mbar_wait(bar(C::B_DS), ph, abort_flag, p.err, kErrTimeoutMma)) break;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint64_t a = desc_add(q_mn, 2 * h * C::QSUB);
          const uint32_t dst = tmem + C::COL_DK + 64 * h;
          if (s == 0)
            mma_ss_k<ID_T, 0>(dst, a, ds_mn);
          else
            mma_ss_k<ID_T, 1>(dst, a, ds_mn);
#pragma unroll
          for (int kq = 1; kq < 8; ++kq)
            mma_ss_k<ID_T, 1>(dst, desc_add(a, kq * 2048), desc_add(ds_mn, kq * 2048));
          mma_commit(bar(C::B_QEMPTY + h));  // Q half h is no longer read
        }
        mma_commit(bar(C::B_DSFREE));
        if (s == n_steps - 1) mma_commit(bar(C::B_FINAL));
      }
      if (*abort_flag) {
        mma_commit(bar(C::B_DRAIN));
        mbar_wait_timed(bar(C::B_DRAIN), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ query rows
    // L and D come from the grid before (the row-dot pass writes D).
    grid_dependency_wait();
    const int wq = warp & 3, g = warp >> 2;
    const int row = wq * 32 + static_cast<int>(threadIdx.x & 31);
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int kbase = jt * C::BK + 32 * g;  // first key of this warp's half of the tile
    const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
    // L and D of this thread's row at step s, loaded one step ahead from an
    // index that is always valid and left as loaded until the step that uses
    // them forms -L log2e and -D (dead rows: -L = -inf so P = 0).
    auto load_ld = [&](int s, float& l, float& dd, bool& live) {
      int bhq, it;
      step_coords(s, bhq, it);
      const int q = it * C::BQ + row;
      live = q < p.N;
      const size_t idx = static_cast<size_t>(bhq) * p.N + (live ? q : 0);
      l = p.lse[idx];
      dd = p.Dvec[idx];
    };
    float l_cur = 0.0f, d_cur = 0.0f;
    bool live_cur = false;
    if (n_steps > 0) load_ld(0, l_cur, d_cur, live_cur);
    bool ok = true;
    for (int s = 0; s < n_steps; ++s) {
      const uint32_t ph = s & 1;
      int bhq, it;
      step_coords(s, bhq, it);
      const int q = it * C::BQ + row;
      const float nl_cur = live_cur ? -l_cur * kLog2e : -INFINITY;
      const float nd_cur = live_cur ? -d_cur : 0.0f;
      const uint64_t nl2 = f2_pack(nl_cur, nl_cur), nd2 = f2_pack(nd_cur, nd_cur);
      if (s + 1 < n_steps) load_ld(s + 1, l_cur, d_cur, live_cur);  // used at the next step
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::B_S), ph, abort_flag, p.err, kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(tmem + lane_off + C::COL_S + 32 * g, sv);
      // Masking only where a key of this warp's half lies past N or past a
      // row of the warp (the diagonal tile); warp-uniform.
      const bool masked =
          __any_sync(0xffffffffu, kbase + 31 >= p.N || (CAUSAL && kbase + 31 > q));
      tmem_wait_ld();
      float pv[32];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * u]), __uint_as_float(sv[2 * u + 1])), c2,
                         nl2),
                  pv[2 * u], pv[2 * u + 1]);
        pv[2 * u] = ex2_approx(pv[2 * u]);
        pv[2 * u + 1] = ex2_approx(pv[2 * u + 1]);
      }
      if (masked) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (kbase + e >= p.N || (CAUSAL && kbase + e > q)) pv[e] = 0.0f;
      }
      uint32_t pk[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) pk[u] = pack_bf16x2(pv[2 * u], pv[2 * u + 1]);
      // The P buffer is free once dV^T of the step before has read it.
      if (s > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_PFREE), (s - 1) & 1, abort_flag, p.err,
                                               kErrTimeoutSoftmax));
        if (!ok) break;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
        st_shared_v4(sP + sw128(row, 4 * g + c), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                     pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_warp(bar(C::B_P));
      // dS = P o (dP - D)
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::B_DP), ph, abort_flag, p.err, kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      uint32_t dpv[32];
      tmem_ld32(tmem + lane_off + C::COL_DP + 32 * g, dpv);
      tmem_wait_ld();
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        float d0, d1;
        f2_unpack(f2_mul(f2_pack(pv[2 * u], pv[2 * u + 1]),
                         f2_add(f2_pack(__uint_as_float(dpv[2 * u]),
                                        __uint_as_float(dpv[2 * u + 1])),
                                nd2)),
                  d0, d1);
        pk[u] = pack_bf16x2(d0, d1);
      }
      if (s > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DSFREE), (s - 1) & 1, abort_flag, p.err,
                                               kErrTimeoutSoftmax));
        if (!ok) break;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
        st_shared_v4(sDS + sw128(row, 4 * g + c), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                     pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_warp(bar(C::B_DS));
    }
    // ---- epilogue, once every product has completed: warpgroup 0 writes dV,
    // warpgroup 1 dK (times scale).  Lane l of warp w holds head-dimension
    // column 128 h + 32 (w % 4) + l of a half h for the tile's 64 keys.
    if (ok && n_steps > 0)
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::B_FINAL), 0, abort_flag, p.err, kErrTimeoutEpilogue));
    if (ok) {
      tc_fence_after();
      const float mul = g == 0 ? 1.0f : p.scale;
      __nv_bfloat16* out = g == 0 ? p.dv : p.dk;
      const uint32_t col0 = g == 0 ? C::COL_DV : C::COL_DK;
      const int lane = static_cast<int>(threadIdx.x & 31);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const int dcol = 128 * h + 32 * wq + lane;
#pragma unroll 1
        for (int kc = 0; kc < 2; ++kc) {
          uint32_t r[32];
          if (n_steps > 0) {
            tmem_ld32(tmem + lane_off + col0 + 64 * h + 32 * kc, r);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = 0u;  // no query sees these keys
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int key = jt * C::BK + 32 * kc + e;
            if (key < p.N)
              out[(static_cast<size_t>(kvz) * p.N + key) * C::D + dcol] =
                  __float2bfloat16_rn(__uint_as_float(r[e]) * mul);
          }
        }
      }
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

template <bool CAUSAL>
cudaError_t launch_kv256_t(const BwdMaps& m, const float* lse, const float* Dv, void* dk,
                           void* dv, const AttnShape& s, uint32_t* err, cudaStream_t stream) {
  using C = Kv256Cfg;
  auto kern = fa_bwd256_kv_kernel<CAUSAL>;
  cudaError_t e = set_smem_limit_once<fa_bwd256_kv_kernel<CAUSAL>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  Kv256Params p;
  p.lse = lse;
  p.Dvec = Dv;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.N = s.N;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.G = s.Hq / s.Hkv;
  p.n_qtiles = (s.N + C::BQ - 1) / C::BQ;
  p.n_ktiles = (s.N + C::BK - 1) / C::BK;
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.err = err;
  const long long grid = static_cast<long long>(p.n_ktiles) * s.B * s.Hkv;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_dependent(kern, dim3(static_cast<unsigned>(grid)), dim3(C::THREADS),
                          C::SMEM_BYTES, stream, m.q, m.k, m.v, m.dO, p);
}

}  // namespace

cudaError_t launch_backward_d256_kv(const BwdMaps& m, const float* lse, const float* Dv, void* dk,
                                    void* dv, const AttnShape& s, uint32_t* err,
                                    cudaStream_t stream) {
  return s.causal ? launch_kv256_t<true>(m, lse, Dv, dk, dv, s, err, stream)
                  : launch_kv256_t<false>(m, lse, Dv, dk, dv, s, err, stream);
}

}  // namespace fa
