// dQ kernel of the deterministic backward pass on sm_103a.
//
// "L'attention fusionnee", section "La passe arriere : recalculer plutot que
// garder", describes two kernels instead of one: one for dK and dV, and one
// for dQ that walks the key tiles in the forward pass's order.  It recomputes
// S and dP (three products more than the single kernel) but needs no atomic
// addition, so the result does not depend on the order in which the GPU runs
// its blocks and repeated runs give identical bits.  This is the dQ kernel.
//
// One CTA owns 128 query rows of one (batch, query head), like the forward:
//   S_j  = Q K_j^T            tcgen05.mma, operands in shared memory
//   dP_j = dO V_j^T           tcgen05.mma
//   P    = exp2(S scale log2e - L log2e), dS = P o (dP - D)   threads
//   dQ  += dS K_j             tcgen05.mma, A = dS (bf16) from tensor memory
// and at the end dq = bf16(scale dQ).  Under the causal mask query tile i
// visits key tiles 0..i only (tiles wholly in the future are skipped).
//
// Pipeline: S_j goes to one of two tensor-memory S buffers (j mod 2) and dP_j
// to a single dP buffer.  The row warps load S_j and dP_j, release the dP
// buffer at once (dP_{j+1} is computed while they work), turn the values into
// dS_j and write it as bf16 over the S columns they have read; then dQ_j
// reads it and S_{j+2} takes the buffer.  S_{j+1} was computed one tile
// ahead, so the threads and the tensor core work at the same time.  No row
// reduction is needed (P comes from the saved L), so each query row is split
// between two warps, 64 key columns each.
//
// Warps: 0-7 query rows (warp w: rows 32 (w % 4).., key columns KH (w / 4)..
// with KH = BN / 2), 8 TMA producer, 9 MMA issuer and tensor-memory owner.
// Tensor memory: S buffers [0,BN) and [BN,2BN) (dS as bf16 pairs at columns
// KH g.. over the S columns warp group g read), dP [2BN,3BN), dQ [COL_DQ,
// COL_DQ + DP).  Keys come in tiles of BN = 128, or of 64 at D = 256, where
// the 256-column fp32 dQ leaves room for 64-column S and dP buffers only.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Head dimension D in {64, 96, 128, 256}; tiles are DP = D rounded up to a
// multiple of 64 columns wide (zero-filled past D), S and dP contract over the
// D real columns and dQ runs at N = D.
template <int D>
struct DqCfg {
  static constexpr int DP = (D + 63) / 64 * 64;  // padded head dimension
  static constexpr int BM = 128;                 // query rows per CTA
  static constexpr int BN = (D == 256) ? 64 : 128;  // keys per tile
  static constexpr int KH = BN / 2;              // key columns per row warp
  static constexpr int SUB = DP / 64;
  static constexpr int QSUB = 128 * 128;         // 128 query rows x 64 bf16
  static constexpr int KSUB = BN * 128;          // BN key rows x 64 bf16
  static constexpr int QTILE = SUB * QSUB;
  static constexpr int KTILE = SUB * KSUB;
  // K_j is read by S_j and dQ_j, and S_{j+2} is issued right after dQ_j:
  // three K stages let K_{j+2} arrive while K_j and K_{j+1} are in use.
  // V_j is read by dP_j only.  At D = 256 (64 KB Q and dO tiles) two K
  // stages and one V stage are what fits.
  static constexpr int NSK = (D == 64) ? 4 : (D == 256 ? 2 : 3);
  static constexpr int NSV = (D == 64) ? 4 : (D == 256 ? 1 : 2);
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + QTILE;
  static constexpr int OFF_K = OFF_DO + QTILE;
  static constexpr int OFF_V = OFF_K + NSK * KTILE;
  static constexpr int OFF_BAR = OFF_V + NSV * KTILE;
  static constexpr int B_QD = 0;
  static constexpr int B_KFULL = 1;                // [NSK]
  static constexpr int B_KEMPTY = B_KFULL + NSK;   // [NSK]
  static constexpr int B_VFULL = B_KEMPTY + NSK;   // [NSV]
  static constexpr int B_VEMPTY = B_VFULL + NSV;   // [NSV]
  static constexpr int B_SFULL = B_VEMPTY + NSV;   // [2] S_j in S buffer j % 2
  static constexpr int B_DPFULL = B_SFULL + 2;     // dP_j in the dP buffer
  static constexpr int B_DPFREE = B_DPFULL + 1;    // dP_j read by every row warp (8 arrivals)
  static constexpr int B_DSREADY = B_DPFREE + 1;   // [2] dS_j in S buffer j % 2 (8 arrivals)
  static constexpr int B_DQDONE = B_DSREADY + 2;   // every dQ MMA done (completes once)
  static constexpr int B_DRAIN = B_DQDONE + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 320;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0, COL_DP = 2 * BN;  // S buffer b at COL_S + BN b
  static constexpr uint32_t COL_DQ = (D == 256) ? 256 : 384;
  static_assert(COL_DQ + DP <= TMEM_COLS, "tensor memory");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct DqParams {
  const float* lse;
  const float* Dvec;
  __nv_bfloat16* dq;
  int N, Hq, G, n_qtiles, n_ktiles, n_heads, heads_per_group;
  float scale;
  float scale_log2;
  uint32_t* err;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(320, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmdO, const DqParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  // Same launch order as the forward: groups of heads, heaviest tiles first.
  const int per_group = p.heads_per_group * p.n_qtiles;
  const int grp = static_cast<int>(blockIdx.x) / per_group;
  const int rem = static_cast<int>(blockIdx.x) - grp * per_group;
  const int in_grp = min(p.heads_per_group, p.n_heads - grp * p.heads_per_group);
  const int qi_ = rem / in_grp;
  const int bh = grp * p.heads_per_group + (rem - qi_ * in_grp);
  const int qt = CAUSAL ? (p.n_qtiles - 1 - qi_) : qi_;
  const int b = bh / p.Hq;
  const int hq = bh - b * p.Hq;
  const int kvz = b * (p.Hq / p.G) + hq / p.G;
  // Under the causal mask the tile's last row qt BM + BM - 1 sees key tiles
  // up to the one holding that position.
  const int n_kv = CAUSAL ? min((qt * C::BM + C::BM - 1) / C::BN + 1, p.n_ktiles) : p.n_ktiles;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_QD), 1);
    for (int s = 0; s < C::NSK; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < C::NSV; ++s) {
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int b2 = 0; b2 < 2; ++b2) {
      mbar_init(bar(C::B_SFULL + b2), 1);
      mbar_init(bar(C::B_DSREADY + b2), 8);
    }
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_DPFREE), 8);
    mbar_init(bar(C::B_DQDONE), 1);
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

  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t sdO = sbase + C::OFF_DO;
  const uint32_t sK = sbase + C::OFF_K;
  const uint32_t sV = sbase + C::OFF_V;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(bar(C::B_QD), 2 * C::QTILE);
#pragma unroll
      for (int s = 0; s < C::SUB; ++s) {
        tma_load_3d(sQ + s * C::QSUB, &tmQ, bar(C::B_QD), 64 * s, qt * C::BM, bh);
        tma_load_3d(sdO + s * C::QSUB, &tmdO, bar(C::B_QD), 64 * s, qt * C::BM, bh);
      }
      // K_j then V_j, in the order the products need them (S_j comes before dP_j).
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int sk = j % C::NSK;
        if (j >= C::NSK && !mbar_wait(bar(C::B_KEMPTY + sk), ((j / C::NSK) - 1) & 1, abort_flag,
                                      p.err, kErrTimeoutLoad))
          break;
        mbar_arrive_expect_tx(bar(C::B_KFULL + sk), C::KTILE);
#pragma unroll
        for (int s = 0; s < C::SUB; ++s)
          tma_load_3d(sK + sk * C::KTILE + s * C::KSUB, &tmK, bar(C::B_KFULL + sk), 64 * s,
                      j * C::BN, kvz);
        k_issued = j + 1;
        const int sv = j % C::NSV;
        if (j >= C::NSV && !mbar_wait(bar(C::B_VEMPTY + sv), ((j / C::NSV) - 1) & 1, abort_flag,
                                      p.err, kErrTimeoutLoad))
          break;
        mbar_arrive_expect_tx(bar(C::B_VFULL + sv), C::KTILE);
#pragma unroll
        for (int s = 0; s < C::SUB; ++s)
          tma_load_3d(sV + sv * C::KTILE + s * C::KSUB, &tmV, bar(C::B_VFULL + sv), 64 * s,
                      j * C::BN, kvz);
        v_issued = j + 1;
      }
      if (*abort_flag) {
        // Let the copies in flight land before the CTA exits.
        mbar_wait_timed(bar(C::B_QD), 0);
        for (int j = max(0, k_issued - C::NSK); j < k_issued; ++j)
          mbar_wait_timed(bar(C::B_KFULL + j % C::NSK), (j / C::NSK) & 1);
        for (int j = max(0, v_issued - C::NSV); j < v_issued; ++j)
          mbar_wait_timed(bar(C::B_VFULL + j % C::NSV), (j / C::NSV) & 1);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t ID_S = idesc_bf16_f32(128, C::BN, false, false);  // S, dP
      constexpr uint32_t ID_Q = idesc_bf16_f32(128, D, false, true);  // dQ (B = K MN-major), N = D
      const uint64_t q_desc = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t do_desc = smem_desc_sw128(sdO, 16, 1024);
      const uint64_t k_kmaj = smem_desc_sw128(sK, 16, 1024);
      const uint64_t v_kmaj = smem_desc_sw128(sV, 16, 1024);
      const uint64_t k_mn = smem_desc_sw128(sK, C::KSUB, 1024);
      bool ok = mbar_wait(bar(C::B_QD), 0, abort_flag, p.err, kErrTimeoutMma);
      // S_j = Q K_j^T into S buffer j % 2.
      auto issue_s = [&](int j) -> bool {
        const int sk = j % C::NSK;
        if (!mbar_wait(bar(C::B_KFULL + sk), (j / C::NSK) & 1, abort_flag, p.err, kErrTimeoutMma))
          return false;
        tc_fence_after();
        const uint32_t dst = tmem + C::COL_S + C::BN * (j & 1);
        const uint64_t kd = desc_add(k_kmaj, sk * C::KTILE);
        mma_ss_k<ID_S, 0>(dst, q_desc, kd);
#pragma unroll
        for (int kk = 1; kk < D / 16; ++kk)
          mma_ss_k<ID_S, 1>(dst, desc_add(q_desc, (kk >> 2) * C::QSUB + (kk & 3) * 32),
                            desc_add(kd, (kk >> 2) * C::KSUB + (kk & 3) * 32));
        mma_commit(bar(C::B_SFULL + (j & 1)));
        return true;
      };
      // dP_j = dO V_j^T into the dP buffer.
      auto issue_dp = [&](int j) -> bool {
        const int sv = j % C::NSV;
        if (!mbar_wait(bar(C::B_VFULL + sv), (j / C::NSV) & 1, abort_flag, p.err, kErrTimeoutMma))
          return false;
        tc_fence_after();
        const uint64_t vd = desc_add(v_kmaj, sv * C::KTILE);
        mma_ss_k<ID_S, 0>(tmem + C::COL_DP, do_desc, vd);
#pragma unroll
        for (int kk = 1; kk < D / 16; ++kk)
          mma_ss_k<ID_S, 1>(tmem + C::COL_DP,
                            desc_add(do_desc, (kk >> 2) * C::QSUB + (kk & 3) * 32),
                            desc_add(vd, (kk >> 2) * C::KSUB + (kk & 3) * 32));
        mma_commit(bar(C::B_DPFULL));
        mma_commit(bar(C::B_VEMPTY + sv));
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok) ok = issue_dp(0);
      if (ok && n_kv > 1) ok = issue_s(1);
      for (int j = 0; ok && j < n_kv; ++j) {
        // dP_{j+1} as soon as the row warps hold dP_j in registers.
        if (j + 1 < n_kv) {
          if (!mbar_wait(bar(C::B_DPFREE), j & 1, abort_flag, p.err, kErrTimeoutMma)) break;
          tc_fence_after();
          if (!issue_dp(j + 1)) break;
        }
        if (!mbar_wait(bar(C::B_DSREADY + (j & 1)), (j >> 1) & 1, abort_flag, p.err,
                       kErrTimeoutMma))
          break;
        tc_fence_after();
        // dQ += dS_j K_j.  dS of keys KH g.. sits packed (bf16 pairs) at
        // columns KH g.. of the S buffer, 16 keys = 8 columns per step; K_j
        // is read MN-major, 16 key rows (2 KB) per step.
        const int sk = j % C::NSK;
        const uint32_t sb = tmem + C::COL_S + C::BN * (j & 1);
        const uint64_t kmn = desc_add(k_mn, sk * C::KTILE);
        constexpr int KPW = C::KH / 16;  // 16-key steps per row warp's columns
        if (j == 0)
          mma_ts_k<ID_Q, 0>(tmem + C::COL_DQ, sb, kmn);
        else
          mma_ts_k<ID_Q, 1>(tmem + C::COL_DQ, sb, kmn);
#pragma unroll
        for (int kk = 1; kk < C::BN / 16; ++kk)
          mma_ts_k<ID_Q, 1>(tmem + C::COL_DQ, sb + (kk / KPW) * C::KH + (kk % KPW) * 8,
                            desc_add(kmn, kk * 2048));
        mma_commit(bar(C::B_KEMPTY + sk));
        // S_{j+2} reuses this S buffer; the products run in issue order, so it
        // overwrites dS_j only after dQ_j has read it.
        if (j + 2 < n_kv && !issue_s(j + 2)) break;
        // Once, after the last tile: a barrier that completed once per tile
        // could not tell its last phase from an earlier one by parity alone.
        if (j == n_kv - 1) mma_commit(bar(C::B_DQDONE));
      }
      if (*abort_flag) {
        mma_commit(bar(C::B_DRAIN));
        mbar_wait_timed(bar(C::B_DRAIN), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ query rows
    // Warp w reads tensor-memory lanes 32 (w % 4) .. +31 (its query rows)
    // and key columns 64 (w / 4) .. +63 of each tile.
    grid_dependency_wait();  // D comes from the row-dot pass, before the dK/dV grid
    const int wq = warp & 3, g = warp >> 2;
    const int row = wq * 32 + static_cast<int>(threadIdx.x & 31);
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int qi = qt * C::BM + row;
    const bool live = qi < p.N;
    const size_t ridx = static_cast<size_t>(bh) * p.N + (live ? qi : 0);
    const float L2 = live ? p.lse[ridx] * kLog2e : INFINITY;  // dead rows: P = 0
    const float Drow = live ? p.Dvec[ridx] : 0.0f;
    const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
    const uint64_t nl2 = f2_pack(-L2, -L2);
    const uint64_t nd2 = f2_pack(-Drow, -Drow);
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SFULL + (j & 1)), (j >> 1) & 1, abort_flag,
                                             p.err, kErrTimeoutSoftmax));
      if (ok)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DPFULL), j & 1, abort_flag, p.err,
                                               kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      const uint32_t scol = C::COL_S + C::BN * (j & 1) + C::KH * g;
      constexpr int KH = C::KH;
      uint32_t sv[KH], dpv[KH];
#pragma unroll
      for (int c = 0; c < KH / 32; ++c) {
        tmem_ld32(tmem + lane_off + scol + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * c]));
        tmem_ld32(tmem + lane_off + C::COL_DP + KH * g + 32 * c,
                  *reinterpret_cast<uint32_t(*)[32]>(&dpv[32 * c]));
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(bar(C::B_DPFREE));
      const int kbase = j * C::BN + KH * g;
      const bool need_mask = (kbase + KH > p.N) || (CAUSAL && kbase + KH - 1 > qt * C::BM);
      uint32_t pk[KH / 2];
      // One copy of the loop with the (warp-uniform) mask and one without: a
      // branch inside the unrolled loop would split it into blocks scheduled
      // one by one (one copy with the branch measured 14 % slower at d = 64).
      auto ds_pass = [&](auto masked_t) {
#pragma unroll
        for (int u = 0; u < KH / 2; ++u) {
          float p0, p1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * u]), __uint_as_float(sv[2 * u + 1])),
                           c2, nl2),
                    p0, p1);
          p0 = ex2_approx(p0);
          p1 = ex2_approx(p1);
          if constexpr (decltype(masked_t)::value) {
            const int key = kbase + 2 * u;
            if (key >= p.N || (CAUSAL && key > qi)) p0 = 0.0f;
            if (key + 1 >= p.N || (CAUSAL && key + 1 > qi)) p1 = 0.0f;
          }
          const uint64_t dd =
              f2_add(f2_pack(__uint_as_float(dpv[2 * u]), __uint_as_float(dpv[2 * u + 1])), nd2);
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p0, p1), dd), d0, d1);
          pk[u] = pack_bf16x2(d0, d1);
        }
      };
      if (need_mask)
        ds_pass(std::true_type{});
      else
        ds_pass(std::false_type{});
      // dS (bf16 pairs) over S columns this warp has already read.
      if constexpr (KH == 64)
        tmem_st32(tmem + lane_off + scol, pk);
      else
        tmem_st16(tmem + lane_off + scol, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(bar(C::B_DSREADY + (j & 1)));
    }
    // ---- epilogue: dq = bf16(scale dQ), one row per thread, 32-column
    // chunks split between the two warps of a row
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DQDONE), 0, abort_flag, p.err,
                                                   kErrTimeoutEpilogue));
    if (ok) {
      tc_fence_after();
      __nv_bfloat16* qrow = p.dq + ridx * D;
#pragma unroll 1
      for (int q4 = g; q4 < D / 32; q4 += 2) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::COL_DQ + q4 * 32, r);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = pack_bf16x2(__uint_as_float(r[2 * u]) * p.scale,
                              __uint_as_float(r[2 * u + 1]) * p.scale);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(qrow + q4 * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
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

template <int D, bool CAUSAL>
cudaError_t launch_dq_t(const BwdMaps& m, const float* lse, const float* Dv, void* dq,
                        const AttnShape& s, uint32_t* err, cudaStream_t stream) {
  using C = DqCfg<D>;
  auto kern = fa_bwd_dq_kernel<D, CAUSAL>;
  cudaError_t e = set_smem_limit_once<fa_bwd_dq_kernel<D, CAUSAL>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  DqParams p;
  p.lse = lse;
  p.Dvec = Dv;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.N = s.N;
  p.Hq = s.Hq;
  p.G = s.Hq / s.Hkv;
  p.n_qtiles = (s.N + C::BM - 1) / C::BM;
  p.n_ktiles = (s.N + C::BN - 1) / C::BN;
  p.n_heads = s.B * s.Hq;
  p.heads_per_group = static_cast<int>(heads_per_group(s.N, D, 2.0, p.G, p.n_heads));
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.err = err;
  const long long grid = static_cast<long long>(p.n_heads) * p.n_qtiles;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_dependent(kern, dim3(static_cast<unsigned>(grid)), dim3(C::THREADS),
                          C::SMEM_BYTES, stream, m.q, m.k, m.v, m.dO, p);
}

}  // namespace

cudaError_t launch_backward_dq(const BwdMaps& m, const float* lse, const float* Dv, void* dq,
                               const AttnShape& s, uint32_t* err, cudaStream_t stream) {
  if (s.d == 64)
    return s.causal ? launch_dq_t<64, true>(m, lse, Dv, dq, s, err, stream)
                    : launch_dq_t<64, false>(m, lse, Dv, dq, s, err, stream);
  if (s.d == 96)
    return s.causal ? launch_dq_t<96, true>(m, lse, Dv, dq, s, err, stream)
                    : launch_dq_t<96, false>(m, lse, Dv, dq, s, err, stream);
  if (s.d == 256)
    return s.causal ? launch_dq_t<256, true>(m, lse, Dv, dq, s, err, stream)
                    : launch_dq_t<256, false>(m, lse, Dv, dq, s, err, stream);
  return s.causal ? launch_dq_t<128, true>(m, lse, Dv, dq, s, err, stream)
                  : launch_dq_t<128, false>(m, lse, Dv, dq, s, err, stream);
}

}  // namespace fa
