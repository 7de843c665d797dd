// Backward pass of exact attention on sm_103a ("L'attention fusionnee",
// section "La passe arriere : recalculer plutot que garder").
//
//   B1  D = rowsum(dO o O), one fp32 value per query row (a memory-bound
//       reduction run before everything else).
//   B2  per key tile: rebuild P from the saved L, then dV, dS, dK, dQ.
//   B3  dQ accumulator (fp32) -> bf16, times scale.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ B1
// TPR threads per row (a power of two, aligned within a warp), each loading
// VPT 16-byte pieces of O and of dO (pieces part, part + TPR, ...); the
// partial sums of a row are combined with warp shuffles.  When `dq_acc` is not
// null the same threads also zero the row of the fp32 dQ accumulator (the
// 32 bytes that match each 16-byte piece), which saves a separate memset.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const uint4* __restrict__ o,
                                                         const uint4* __restrict__ dO,
                                                         float* __restrict__ out, long long rows,
                                                         float4* __restrict__ dq_acc) {
  constexpr int PIECES = D / 8;                   // 16-byte pieces per row: 8, 12, 16 or 32
  constexpr int TPR = (PIECES % 4 == 0 && PIECES % 8 != 0) ? 4 : PIECES;
  constexpr int VPT = PIECES / TPR;
  static_assert(TPR * VPT == PIECES && (TPR & (TPR - 1)) == 0, "row split");
  // Launched as a programmatic dependent: O and dO are read only once the
  // grid before has completed.  The backward's main kernel, launched as this
  // grid's dependent, may then start its own set-up (it reads only the
  // inputs before it waits for this grid, and D and the accumulator after).
  grid_dependency_wait();
  grid_launch_dependents();
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = tid / TPR;
  const int part = static_cast<int>(tid % TPR);
  float acc = 0.0f;
  if (row < rows) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const long long piece = row * PIECES + part + v * TPR;
      const uint4 a = __ldg(o + piece);
      const uint4 g = __ldg(dO + piece);
      if (dq_acc) {
        dq_acc[2 * piece] = make_float4(0.f, 0.f, 0.f, 0.f);
        dq_acc[2 * piece + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const uint32_t av[4] = {a.x, a.y, a.z, a.w};
      const uint32_t gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 af = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[t]));
        const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[t]));
        acc = fmaf(af.x, gf.x, acc);
        acc = fmaf(af.y, gf.y, acc);
      }
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) out[row] = acc;
}

// ------------------------------------------------------------------ B3
__global__ void __launch_bounds__(256) dq_finalize_kernel(const float4* __restrict__ acc,
                                                          uint4* __restrict__ dq, long long n8,
                                                          float scale) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  grid_dependency_wait();  // the accumulator is complete once the main kernel is
  grid_launch_dependents();
  if (i >= n8) return;
  // L2 loads: the accumulator was written by the grid before, which ran
  // while this one was already resident.
  const float4 a = __ldcg(acc + 2 * i);
  const float4 b = __ldcg(acc + 2 * i + 1);
  dq[i] = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                     pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
}


// ------------------------------------------------------------------ B2
//
// One CTA owns one tile of 128 keys of one (batch, key/value head) and keeps
// its dK and dV accumulators in tensor memory while it walks every query
// tile of every query head of the group that sees those keys (FlashAttention-2
// order as "L'attention fusionnee" describes it: one block per key tile,
// dK and dV kept on chip, dQ added to global memory).  Keys sit on the 128
// TMEM lanes, so each softmax thread owns one key row.  Per query tile i:
//
//   S^T  = K_j Q_i^T - L_i / scale    tcgen05.mma, A and B K-major in smem;
//                                     L_i (saved by the forward) enters as one
//                                     more k-step: A = ones, B = -L_i / scale
//                                     as three bf16 terms per query
//   dP^T = V_j dO_i^T - D_i           tcgen05.mma, D_i (from B1) the same way
//   P^T  = exp2(S^T scale log2e)                  threads
//   dS^T = P^T o dP^T                             threads
//   dV  += P^T dO_i                   tcgen05.mma, A = P^T (bf16) from TMEM
//   dK  += dS^T Q_i                   tcgen05.mma, A = dS^T (bf16, K-major smem)
//   dQ_i = dS K_j                     tcgen05.mma, A = the same dS^T buffer read
//                                     MN-major; drained by a TMA reduce-add
//                                     into the fp32 dQ accumulator
// dK is multiplied by scale once at the end; dQ gets its scale in B3.
//
// Warp roles (384 threads): warps 0-3 key rows (P^T, dS^T, the next step's
// -L/scale and -D rows of the extra k-step, epilogue),
// warps 4-7 dQ drain, warp 8 TMA, warp 9 MMA, warps 10-11 idle.  The drain
// warpgroup takes a step's dQ out of TMEM at once (freeing the columns for
// the next dP^T) and reduces it while the key-row warps go on to the next
// step.  Registers: 152 for warps 8-11, 200 key rows, 152 drain
// (128 x (200 + 152 + 152) = 384 x 168, the launch total).
// Tensor memory: dK [0, DP), dV [DP, 2DP), S^T/P^T 128 columns, dP^T 128
// columns, dQ 64 columns after dP^T when D = 64, or in dP^T's columns when
// DP = 128 (DP = D rounded up to a multiple of 64).

// Head dimension D in {96, 128} (64 has its own kernel).  Tiles are DP = 128
// columns wide; for D = 96 the copies zero-fill columns 96..127, S^T and dP^T
// contract over the D real columns, and dV, dK and dQ run at N = D.
template <int D>
struct BwdCfg {
  static constexpr int DP = (D + 63) / 64 * 64;  // padded head dimension
  static constexpr int BK = 128;                // keys per CTA
  static constexpr int BQ = 128;                // queries per step
  static constexpr int SUB = DP / 64;
  static constexpr int SUB_BYTES = 128 * 128;
  static constexpr int TILE = SUB * SUB_BYTES;  // 128 x DP bf16
  // Q has two stages, so that S^T of the next step needs no load; dO has one,
  // released as soon as dV has read it.  dQ leaves through a 16 KB staging
  // tile, one 32 x 32 fp32 box per drain warp, each refilled once that warp's
  // previous reduce has read it.
  static constexpr int NQ = 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;
  static constexpr int OFF_DO = OFF_Q + NQ * TILE;
  static constexpr int OFF_DS = OFF_DO + TILE;    // dS^T: 128 keys x 128 queries bf16
  static constexpr int OFF_STG = OFF_DS + 2 * SUB_BYTES;  // dQ staging: 4 x (32 rows x 32 fp32)
  // Operands of S^T's and dP^T's last k-step: a 128 x 64 bf16 tile in the
  // 128-byte swizzled layout whose 16-column slot 0 holds ones in columns
  // 0-2 of every row (A, one row per key), slot 1 -L/scale and slot 2 -D of
  // the step's queries as three bf16 terms each (B, one row per query).
  static constexpr int OFF_AUG = OFF_STG + SUB_BYTES;
  static constexpr int OFF_BAR = OFF_AUG + SUB_BYTES;
  static constexpr int B_KV = 0;
  static constexpr int B_QFULL = 1;               // [NQ]
  static constexpr int B_QEMPTY = B_QFULL + NQ;   // [NQ]
  static constexpr int B_DOFULL = B_QEMPTY + NQ;
  static constexpr int B_DOEMPTY = B_DOFULL + 1;
  static constexpr int B_S = B_DOEMPTY + 1;       // S^T in TMEM
  static constexpr int B_DP = B_S + 1;            // dP^T in TMEM
  static constexpr int B_P = B_DP + 1;            // P^T in TMEM, S^T read (128 arrivals)
  static constexpr int B_DS = B_P + 1;            // dS^T in smem, dP^T read (128 arrivals)
  static constexpr int B_DQFULL = B_DS + 1;       // dQ in TMEM (dV, dP^T, dQ of the step done)
  static constexpr int B_DQFREE = B_DQFULL + 1;   // dQ columns drained (128 arrivals)
  static constexpr int B_FINAL = B_DQFREE + 1;    // every product issued has completed (once)
  static constexpr int B_DRAIN = B_FINAL + 1;
  static constexpr int B_AUG0 = B_DRAIN + 1;      // step 0's blocks written (128 arrivals)
  static constexpr int NBAR = B_AUG0 + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_DK = 0;
  static constexpr uint32_t COL_DV = DP;
  static constexpr uint32_t COL_S = 2 * DP;
  static constexpr uint32_t COL_DP = 2 * DP + 128;
  static constexpr uint32_t COL_DQ = (D == 64) ? 2 * DP + 256 : COL_DP;
};

struct BwdParams {
  const float* lse;
  const float* Dvec;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int N, Hq, Hkv, G, n_qtiles;
  float scale;
  float scale_log2;
  uint32_t* err;
};

// Byte offset of 16-byte chunk `ch` of row `r` in a 128-byte-swizzled block
// of 128-byte rows (the layout TMA and tcgen05 agree on).
__device__ __forceinline__ uint32_t sw128(int r, int ch) {
  return static_cast<uint32_t>(r * 128 + ((ch ^ (r & 7)) << 4));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// This thread's row of an fp32 TMEM accumulator (D columns from `taddr`)
// times `mul`, as bf16 into `row` (skipped for rows past N).  Warp-collective.
template <int D>
__device__ __forceinline__ void write_rows(uint32_t taddr, __nv_bfloat16* row, float mul,
                                           bool live) {
#pragma unroll
  for (int q4 = 0; q4 < D / 32; ++q4) {
    uint32_t r[32];
    tmem_ld32(taddr + q4 * 32, r);
    tmem_wait_ld();
    uint32_t pk[16];
#pragma unroll
    for (int u = 0; u < 16; ++u)
      pk[u] = pack_bf16x2(__uint_as_float(r[2 * u]) * mul, __uint_as_float(r[2 * u + 1]) * mul);
    if (live) {
      uint4* dst = reinterpret_cast<uint4*>(row + q4 * 32);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
    }
  }
}

// DQ = false builds the dK/dV-only kernel of the deterministic backward.
template <int D, bool CAUSAL, bool DQ>
__global__ void __launch_bounds__(384, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmdQ, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int kvz = blockIdx.x;  // flattened (batch, kv head)
  const int jt = blockIdx.y;   // key tile
  const int b = kvz / p.Hkv;
  const int hkv = kvz - b * p.Hkv;
  const int i0 = CAUSAL ? jt : 0;  // first query tile that sees this key tile
  const int per_head = p.n_qtiles - i0;
  const int n_steps = p.G * per_head;

  const uint32_t sK = sbase + C::OFF_K;
  const uint32_t sV = sbase + C::OFF_V;
  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t sdO = sbase + C::OFF_DO;
  const uint32_t sDS = sbase + C::OFF_DS;
  const uint32_t sSTG = sbase + C::OFF_STG;

  // The producer's lane initialises the barriers and issues the loads of K,
  // V and step 0's Q and dO at once, so that their latency overlaps the
  // tensor-memory allocation and the CTA barrier below.  (K, V, Q and dO are
  // inputs of the backward, which this grid may read before it waits for
  // the grid before it.)
  if (warp == 8 && elect_one()) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    mbar_init(bar(C::B_KV), 1);
    for (int s = 0; s < C::NQ; ++s) {
      mbar_init(bar(C::B_QFULL + s), 1);
      mbar_init(bar(C::B_QEMPTY + s), 1);
    }
    mbar_init(bar(C::B_DOFULL), 1);
    mbar_init(bar(C::B_DOEMPTY), 1);
    mbar_init(bar(C::B_S), 1);
    mbar_init(bar(C::B_DP), 1);
    mbar_init(bar(C::B_P), 128);
    mbar_init(bar(C::B_DS), 128);
    mbar_init(bar(C::B_DQFULL), 1);
    mbar_init(bar(C::B_DQFREE), 128);
    mbar_init(bar(C::B_FINAL), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    mbar_init(bar(C::B_AUG0), 128);
    *abort_flag = 0;
    fence_barrier_init();
    mbar_arrive_expect_tx(bar(C::B_KV), 2 * C::TILE);
#pragma unroll
    for (int s = 0; s < C::SUB; ++s) {
      tma_load_3d(sK + s * C::SUB_BYTES, &tmK, bar(C::B_KV), 64 * s, jt * C::BK, kvz);
      tma_load_3d(sV + s * C::SUB_BYTES, &tmV, bar(C::B_KV), 64 * s, jt * C::BK, kvz);
    }
    if (n_steps > 0) {  // step 0: query head 0 of the group, query tile i0
      const int bhq = b * p.Hq + hkv * p.G;
      mbar_arrive_expect_tx(bar(C::B_QFULL), C::TILE);
      mbar_arrive_expect_tx(bar(C::B_DOFULL), C::TILE);
#pragma unroll
      for (int s = 0; s < C::SUB; ++s) {
        tma_load_3d(sQ + s * C::SUB_BYTES, &tmQ, bar(C::B_QFULL), 64 * s, i0 * C::BQ, bhq);
        tma_load_3d(sdO + s * C::SUB_BYTES, &tmdO, bar(C::B_DOFULL), 64 * s, i0 * C::BQ, bhq);
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

  if (warp >= 8) {
    reg_decrease<152>();
    if (warp == 8) {
      // ------------------------------------------------------------ TMA producer
      if (elect_one()) {
        // Q of step s into stage s % NQ, dO into its single stage; each waits
        // for the step that last used its buffer.  K, V and step 0 were
        // issued before the CTA barrier.
        int q_issued = n_steps > 0 ? 1 : 0, do_issued = q_issued;
        for (int st_i = 1; st_i < n_steps; ++st_i) {
          const int g = st_i / per_head;
          const int it = i0 + (st_i - g * per_head);
          const int bhq = b * p.Hq + hkv * p.G + g;
          const int qs = st_i % C::NQ;
          if (st_i >= C::NQ && !mbar_wait(bar(C::B_QEMPTY + qs), ((st_i / C::NQ) - 1) & 1,
                                          abort_flag, p.err, kErrTimeoutLoad))
            break;
          mbar_arrive_expect_tx(bar(C::B_QFULL + qs), C::TILE);
  #pragma unroll
          for (int s = 0; s < C::SUB; ++s)
            tma_load_3d(sQ + qs * C::TILE + s * C::SUB_BYTES, &tmQ, bar(C::B_QFULL + qs), 64 * s,
                        it * C::BQ, bhq);
          q_issued = st_i + 1;
          if (st_i >= 1 && !mbar_wait(bar(C::B_DOEMPTY), (st_i - 1) & 1, abort_flag, p.err,
                                      kErrTimeoutLoad))
            break;
          mbar_arrive_expect_tx(bar(C::B_DOFULL), C::TILE);
  #pragma unroll
          for (int s = 0; s < C::SUB; ++s)
            tma_load_3d(sdO + s * C::SUB_BYTES, &tmdO, bar(C::B_DOFULL), 64 * s, it * C::BQ, bhq);
          do_issued = st_i + 1;
        }
        if (*abort_flag) {
          mbar_wait_timed(bar(C::B_KV), 0);
          for (int s2 = max(0, q_issued - C::NQ); s2 < q_issued; ++s2)
            mbar_wait_timed(bar(C::B_QFULL + s2 % C::NQ), (s2 / C::NQ) & 1);
          if (do_issued > 0) mbar_wait_timed(bar(C::B_DOFULL), (do_issued - 1) & 1);
        }
      }
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      if (elect_one()) {
        constexpr uint32_t id_ss = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
        // dV, dK and dQ run at N = D (a multiple of 16): at D = 96 the padded
        // columns of their accumulators are neither computed nor read.
        constexpr uint32_t id_kd = idesc_bf16_f32(128, D, false, true);  // dV, dK
        constexpr uint32_t id_q = idesc_bf16_f32(128, D, true, true);    // dQ
        bool ok = mbar_wait(bar(C::B_KV), 0, abort_flag, p.err, kErrTimeoutMma) &&
                  mbar_wait(bar(C::B_AUG0), 0, abort_flag, p.err, kErrTimeoutMma);
        const uint64_t aug_a = smem_desc_sw128(sbase + C::OFF_AUG, 16, 1024);  // ones, slot 0
        // S^T of step s (Q_s in stage s % NQ) into the S^T columns.
        auto issue_s = [&](int s) -> bool {
          const int qs = s % C::NQ;
          if (!mbar_wait(bar(C::B_QFULL + qs), (s / C::NQ) & 1, abort_flag, p.err, kErrTimeoutMma))
            return false;
          tc_fence_after();
          const uint32_t q_st = sQ + qs * C::TILE;
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::SUB_BYTES + (kk & 3) * 32;
            mma_ss(tmem + C::COL_S, smem_desc_sw128(sK + off, 16, 1024),
                   smem_desc_sw128(q_st + off, 16, 1024), id_ss, kk > 0 ? 1u : 0u);
          }
          mma_ss(tmem + C::COL_S, aug_a, desc_add(aug_a, 32), id_ss, 1u);  // - L / scale
          mma_commit(bar(C::B_S));
          return true;
        };
        // dP^T of step s into the dP^T columns, which hold dQ of step s - 1
        // until the drain has taken it.
        auto issue_dp = [&](int s) -> bool {
          if (s > 0 &&
              !mbar_wait(bar(C::B_DQFREE), (s - 1) & 1, abort_flag, p.err, kErrTimeoutMma))
            return false;
          if (!mbar_wait(bar(C::B_DOFULL), s & 1, abort_flag, p.err, kErrTimeoutMma)) return false;
          tc_fence_after();
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::SUB_BYTES + (kk & 3) * 32;
            mma_ss(tmem + C::COL_DP, smem_desc_sw128(sV + off, 16, 1024),
                   smem_desc_sw128(sdO + off, 16, 1024), id_ss, kk > 0 ? 1u : 0u);
          }
          mma_ss(tmem + C::COL_DP, aug_a, desc_add(aug_a, 64), id_ss, 1u);  // - D
          mma_commit(bar(C::B_DP));
          return true;
        };
        if (ok && n_steps > 0) ok = issue_s(0) && issue_dp(0);
        // Per step: dV once the threads have written P^T, then the next S^T
        // over it (the tensor pipe runs in issue order); dK and dQ once they
        // have written dS^T, then the next dP^T once the drain has taken dQ.
        // The threads compute dS^T while dV and the next S^T run, and the
        // next step's P^T while dK, dQ, the drain and the next dP^T run.
        for (int s = 0; ok && s < n_steps; ++s) {
          const int qs = s % C::NQ;
          const uint32_t q_st = sQ + qs * C::TILE;
          const uint32_t do_st = sdO;
          if (!mbar_wait(bar(C::B_P), s & 1, abort_flag, p.err, kErrTimeoutMma)) break;
          tc_fence_after();
          // dV += P^T dO_i   (A = P^T in TMEM: 16 queries = 8 packed columns per step)
  #pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C::COL_DV, tmem + C::COL_S + kk * 8,
                   smem_desc_sw128(do_st + kk * 2048, C::SUB_BYTES, 1024), id_kd,
                   (s > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(C::B_DOEMPTY));  // dO_i is not read after dV
          if (s + 1 < n_steps && !issue_s(s + 1)) break;
          if (!mbar_wait(bar(C::B_DS), s & 1, abort_flag, p.err, kErrTimeoutMma)) break;
          tc_fence_after();
          // dQ_i = dS K_j first (A = dS: the dS^T buffer read MN-major; B = K_j
          // MN-major), so that the drain takes it while dK runs.
  #pragma unroll
          for (int kk = 0; kk < (DQ ? 8 : 0); ++kk)
            mma_ss(tmem + C::COL_DQ, smem_desc_sw128(sDS + kk * 2048, C::SUB_BYTES, 1024),
                   smem_desc_sw128(sK + kk * 2048, C::SUB_BYTES, 1024), id_q, kk > 0 ? 1u : 0u);
          mma_commit(bar(C::B_DQFULL));
          // dK += dS^T Q_i   (A = dS^T K-major: queries contiguous per key row)
  #pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * C::SUB_BYTES + (kk & 3) * 32;
            mma_ss(tmem + C::COL_DK, smem_desc_sw128(sDS + off, 16, 1024),
                   smem_desc_sw128(q_st + kk * 2048, C::SUB_BYTES, 1024), id_kd,
                   (s > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(C::B_QEMPTY + qs));  // Q_i is not read after dK
          // Once, after the last step: every product has completed (the dK
          // accumulator is final).
          if (s == n_steps - 1) mma_commit(bar(C::B_FINAL));
          if (s + 1 < n_steps && !issue_dp(s + 1)) break;
        }
        if (*abort_flag) {
          mma_commit(bar(C::B_DRAIN));
          mbar_wait_timed(bar(C::B_DRAIN), 0);
        }
      }
    }
  } else if (warp < 4) {
    reg_increase<200>();
    // ------------------------------------------------------------ key rows
    // L and D are read only once the row-dot pass (the grid before this one)
    // has completed.
    grid_dependency_wait();
    const int t = threadIdx.x;  // key row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int key = jt * C::BK + t;
    const bool key_live = key < p.N;
    const float c = p.scale_log2;
    bool ok = true;
    // L and D of query row t of step s, loaded during the step before from
    // an index that is always valid (row 0 for rows past N), and left as
    // loaded until this thread writes them as row t of the extra k-step's
    // B operands (-L/scale and -D; dead rows -inf, so P = 0, and 0).
    // Nothing then waits for the loads within the step that issues them.
    auto load_ld = [&](int s, float& lv, float& dv, bool& live) {
      const int g = s / per_head;
      const int qrow = (i0 + (s - g * per_head)) * C::BQ + t;
      live = qrow < p.N;
      const size_t idx = static_cast<size_t>(b * p.Hq + hkv * p.G + g) * p.N + (live ? qrow : 0);
      lv = p.lse[idx];
      dv = p.Dvec[idx];
    };
    float l_cur = 0.0f, d_cur = 0.0f;
    bool live_cur = false;
    if (n_steps > 0) load_ld(0, l_cur, d_cur, live_cur);
    // Row t of the extra k-step's tile: v as hi + mid + lo (bf16) in
    // columns 0-2 of 16-column slot `slot`.
    const uint32_t sAug = sbase + C::OFF_AUG;
    auto write_aug = [&](int slot, float v) {
      float hi = v, mid = 0.0f, lo = 0.0f;
      if (isfinite(v)) {
        hi = __bfloat162float(__float2bfloat16_rn(v));
        const float r1 = v - hi;
        mid = __bfloat162float(__float2bfloat16_rn(r1));
        lo = r1 - mid;
      }
      st_shared_v4(sAug + sw128(t, 2 * slot), pack_bf16x2(hi, mid), pack_bf16x2(lo, 0.0f), 0u,
                   0u);
      st_shared_v4(sAug + sw128(t, 2 * slot + 1), 0u, 0u, 0u, 0u);
    };
    // Ones in slot 0 (bf16 1.0 = 0x3f80) and step 0's -L/scale and -D.
    st_shared_v4(sAug + sw128(t, 0), 0x3f803f80u, 0x3f80u, 0u, 0u);
    st_shared_v4(sAug + sw128(t, 1), 0u, 0u, 0u, 0u);
    if (n_steps > 0) {
      write_aug(1, live_cur ? -__fdiv_rn(l_cur, p.scale) : -INFINITY);
      write_aug(2, live_cur ? -d_cur : 0.0f);
    }
    fence_proxy_async_smem();
    mbar_arrive(bar(C::B_AUG0));
    // Step s + 1's dS^T overwrites step s's in shared memory: it is written
    // once dP^T of step s + 1 is in, which is computed only after the drain
    // has taken step s's dQ, so every product of step s (the ones reading
    // dS^T too) has completed.
    for (int s = 0; s < n_steps; ++s) {
      const int g = s / per_head;
      const int it = i0 + (s - g * per_head);
      const int q0 = it * C::BQ;
      if (s + 1 < n_steps) load_ld(s + 1, l_cur, d_cur, live_cur);  // written during this step
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::B_S), s & 1, abort_flag, p.err, kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      // Masking is needed only on the diagonal tile and for keys past N.
      const bool masked = __any_sync(0xffffffffu, (CAUSAL && it == jt) || !key_live);
      const uint64_t c2 = f2_pack(c, c);
      // ---- P^T = exp2(S^T c - L log2e), kept as packed bf16 for dS^T.
      // Chunk cc + 1 (32 query columns) is loaded while chunk cc is
      // computed; P^T of chunk cc goes to columns 16cc.., below the S^T
      // columns 32(cc + 1).. being loaded.
      uint32_t pk[64];
      // Two copies of the pass, with and without the mask (warp-uniform):
      // a branch inside the unrolled loop would split it into blocks that
      // the compiler schedules one by one, and each chunk's exponentials
      // would then wait out the full load / multiply-add / exp2 latency in
      // turn (one copy with the branch measured 10-13 % slower at d = 128 and 96).
      auto p_pass = [&](auto masked_t) {
        constexpr bool MASKED = decltype(masked_t)::value;
        uint32_t sv2[2][32];
        tmem_ld32(tmem + lane_off + C::COL_S, sv2[0]);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (cc + 1 < 4) tmem_ld32(tmem + lane_off + C::COL_S + (cc + 1) * 32, sv2[(cc + 1) & 1]);
          const uint32_t(&sv)[32] = sv2[cc & 1];
#pragma unroll
          for (int u4 = 0; u4 < 8; ++u4) {
            float pv[4];
            f2_unpack(f2_mul(f2_pack(__uint_as_float(sv[4 * u4]), __uint_as_float(sv[4 * u4 + 1])),
                             c2),
                      pv[0], pv[1]);
            f2_unpack(
                f2_mul(f2_pack(__uint_as_float(sv[4 * u4 + 2]), __uint_as_float(sv[4 * u4 + 3])),
                       c2),
                pv[2], pv[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) pv[e] = ex2_approx(pv[e]);
            if constexpr (MASKED) {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (!key_live || (CAUSAL && key > q0 + cc * 32 + u4 * 4 + e)) pv[e] = 0.0f;
            }
            pk[cc * 16 + 2 * u4] = pack_bf16x2(pv[0], pv[1]);
            pk[cc * 16 + 2 * u4 + 1] = pack_bf16x2(pv[2], pv[3]);
          }
          tmem_st16(tmem + lane_off + C::COL_S + cc * 16,
                    *reinterpret_cast<const uint32_t(*)[16]>(&pk[cc * 16]));
          if (cc + 1 < 4) tmem_wait_ld();
        }
      };
      if (masked)
        p_pass(std::true_type{});
      else
        p_pass(std::false_type{});
      // S^T of this step has been read: the next step's -L/scale goes into slot 1.
      if (s + 1 < n_steps) {
        write_aug(1, live_cur ? -__fdiv_rn(l_cur, p.scale) : -INFINITY);
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::B_P));
      // ---- dS^T = P^T o (dP^T - D) from the bf16 P^T (as the dV product
      // uses it), into the dS^T buffer in shared memory.
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::B_DP), s & 1, abort_flag, p.err, kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t dpv2[2][32];
        tmem_ld32(tmem + lane_off + C::COL_DP, dpv2[0]);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (cc + 1 < 4)
            tmem_ld32(tmem + lane_off + C::COL_DP + (cc + 1) * 32, dpv2[(cc + 1) & 1]);
          const uint32_t(&dpv)[32] = dpv2[cc & 1];
          uint32_t dk16[16];
#pragma unroll
          for (int u4 = 0; u4 < 8; ++u4) {
            const __nv_bfloat162 pa =
                *reinterpret_cast<const __nv_bfloat162*>(&pk[cc * 16 + 2 * u4]);
            const __nv_bfloat162 pb =
                *reinterpret_cast<const __nv_bfloat162*>(&pk[cc * 16 + 2 * u4 + 1]);
            const float2 p01 = __bfloat1622float2(pa);
            const float2 p23 = __bfloat1622float2(pb);
            const uint64_t ds01 =
                f2_mul(f2_pack(p01.x, p01.y),
                       f2_pack(__uint_as_float(dpv[4 * u4]), __uint_as_float(dpv[4 * u4 + 1])));
            const uint64_t ds23 = f2_mul(
                f2_pack(p23.x, p23.y),
                f2_pack(__uint_as_float(dpv[4 * u4 + 2]), __uint_as_float(dpv[4 * u4 + 3])));
            float dsv[4];
            f2_unpack(ds01, dsv[0], dsv[1]);
            f2_unpack(ds23, dsv[2], dsv[3]);
            dk16[2 * u4] = pack_bf16x2(dsv[0], dsv[1]);
            dk16[2 * u4 + 1] = pack_bf16x2(dsv[2], dsv[3]);
          }
          // dS^T row `t`, queries cc*32 .. cc*32+31: 4 chunks of 8 in block cc/2.
          const uint32_t blk = sDS + (cc >> 1) * C::SUB_BYTES;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            st_shared_v4(blk + sw128(t, (cc & 1) * 4 + q4), dk16[4 * q4], dk16[4 * q4 + 1],
                         dk16[4 * q4 + 2], dk16[4 * q4 + 3]);
          if (cc + 1 < 4) tmem_wait_ld();
        }
      }
      // dP^T of this step has been read: the next step's -D goes into slot 2.
      if (s + 1 < n_steps) write_aug(2, live_cur ? -d_cur : 0.0f);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_DS));
    }
    // ---- epilogue: dK (times scale) and dV, one key row per thread, once
    // every product has completed.
    if (ok && n_steps > 0)
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::B_FINAL), 0, abort_flag, p.err, kErrTimeoutEpilogue));
    if (ok) {
      // dK (times scale); the drain warpgroup writes dV meanwhile.
      tc_fence_after();
      write_rows<D>(tmem + lane_off + C::COL_DK,
                    p.dk + (static_cast<size_t>(kvz) * p.N + (key_live ? key : 0)) * D, p.scale,
                    key_live);
    }
  } else {
    reg_decrease<152>();
    // ------------------------------------------------------------ dQ drain
    // dQ of step s sits in dP^T's columns: take all of it into registers,
    // hand the columns back (the next dP^T may be computed), then reduce it
    // into the fp32 accumulator, D / 32 boxes of 32 columns.  Each warp
    // stages its own 32 rows (4 KB of the staging tile) and its lane 0
    // issues the reduce of that 32 x 32 box, so no warp waits for another;
    // a warp refills its slice once its own previous reduce has read it.
    // The accumulator was zeroed by the row-dot pass (the grid before).
    grid_dependency_wait();
    const int t = threadIdx.x & 127;  // query row of the step's tile
    const int wq = warp & 3;
    const int r = t & 31;             // row within this warp's box
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t sW = sSTG + wq * 4096;
    bool ok = true;
    constexpr int kBoxes = D / 32;
    for (int s = 0; s < n_steps; ++s) {
      const int g = s / per_head;
      const int it = i0 + (s - g * per_head);
      const int bhq = b * p.Hq + hkv * p.G + g;
      const int y0 = it * C::BQ + 32 * wq;  // first query row of this warp's box
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::B_DQFULL), s & 1, abort_flag, p.err, kErrTimeoutOther));
      if (!ok) break;
      tc_fence_after();
      uint32_t dqv[DQ ? kBoxes : 1][32];
      if (DQ) {
#pragma unroll
        for (int x = 0; x < kBoxes; ++x) tmem_ld32(tmem + lane_off + C::COL_DQ + x * 32, dqv[x]);
        tmem_wait_ld();
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_DQFREE));  // dP^T's columns may be overwritten now
      // Rows at or past N are not reduced (a box starting there is skipped).
      const bool box_live = y0 < p.N;
#pragma unroll
      for (int x = 0; x < (DQ ? kBoxes : 0); ++x) {
        if (r == 0) bulk_wait_group_read0();  // this warp's slice is free again
        __syncwarp();
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          st_shared_v4(sW + sw128(r, ch), dqv[x][4 * ch], dqv[x][4 * ch + 1], dqv[x][4 * ch + 2],
                       dqv[x][4 * ch + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (r == 0 && box_live) {
          tma_reduce_add_3d(&tmdQ, sW, x * 32, y0, bhq);
          bulk_commit_group();
        }
      }
    }
    // dV, once the last step's products have completed (its dQ commit, which
    // the loop waited for, covers them); the key-row warpgroup writes dK.
    if (ok && n_steps > 0) {
      tc_fence_after();
      const int vkey = jt * C::BK + t;  // lane t of this warp's quarter is key row t
      const bool vlive = vkey < p.N;
      write_rows<D>(tmem + lane_off + C::COL_DV,
                    p.dv + (static_cast<size_t>(kvz) * p.N + (vlive ? vkey : 0)) * D, 1.0f,
                    vlive);
    }
    // Only the staging tile's reads must be over before the CTA's shared
    // memory is released; the reduces' writes complete on their own, and the
    // dQ finalisation reads the accumulator only after this grid has completed.
    if (r == 0) bulk_wait_group_read0();
    __syncwarp();
    grid_launch_dependents();  // the dQ finalisation may be scheduled
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

}  // namespace

cudaError_t launch_preprocess(const void* o, const void* dO, float* Dout, long long rows, int d,
                              cudaStream_t stream, float* zero_acc) {
  float4* acc = reinterpret_cast<float4*>(zero_acc);
  const long long threads = rows * (d == 96 ? 4 : d / 8);  // threads per row as in the kernel
  const long long blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(blocks)), block(256);
  const uint4* o4 = static_cast<const uint4*>(o);
  const uint4* dO4 = static_cast<const uint4*>(dO);
  if (d == 64)
    return launch_dependent(preprocess_kernel<64>, grid, block, 0, stream, o4, dO4, Dout, rows,
                            acc);
  if (d == 96)
    return launch_dependent(preprocess_kernel<96>, grid, block, 0, stream, o4, dO4, Dout, rows,
                            acc);
  if (d == 256)
    return launch_dependent(preprocess_kernel<256>, grid, block, 0, stream, o4, dO4, Dout, rows,
                            acc);
  return launch_dependent(preprocess_kernel<128>, grid, block, 0, stream, o4, dO4, Dout, rows, acc);
}

cudaError_t launch_dq_finalize(const float* dq_acc, void* dq, long long n, float scale,
                               cudaStream_t stream) {
  const long long n8 = n / 8;  // n = rows x d, a multiple of 32
  const long long blocks = (n8 + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_dependent(dq_finalize_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                          stream, reinterpret_cast<const float4*>(dq_acc),
                          static_cast<uint4*>(dq), n8, scale);
}

template <int D, bool CAUSAL, bool DQ>
cudaError_t launch_bwd_t(const BwdMaps& m, const float* lse, const float* Dv, void* dk, void* dv,
                         const AttnShape& s, uint32_t* err, cudaStream_t stream) {
  using C = BwdCfg<D>;
  auto kern = fa_bwd_kernel<D, CAUSAL, DQ>;
  cudaError_t e = set_smem_limit_once<fa_bwd_kernel<D, CAUSAL, DQ>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  BwdParams p;
  p.lse = lse;
  p.Dvec = Dv;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.N = s.N;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.G = s.Hq / s.Hkv;
  p.n_qtiles = (s.N + C::BQ - 1) / C::BQ;
  p.scale = s.scale;
  p.scale_log2 = s.scale * kLog2e;
  p.err = err;
  const int n_ktiles = (s.N + C::BK - 1) / C::BK;
  dim3 grid(static_cast<unsigned>(s.B * s.Hkv), static_cast<unsigned>(n_ktiles));
  return launch_dependent(kern, grid, dim3(C::THREADS), C::SMEM_BYTES, stream, m.q, m.k, m.v,
                          m.dO, m.dq_acc32, p);
}

cudaError_t launch_backward(const BwdMaps& m, const float* lse, const float* Dv, float*, void* dk,
                            void* dv, const AttnShape& s, uint32_t* err, cudaStream_t stream,
                            bool with_dq) {
  if (s.d == 64) return launch_backward_d64(m, lse, Dv, dk, dv, s, err, stream, with_dq);
  if (s.d == 96) {
    if (with_dq)
      return s.causal ? launch_bwd_t<96, true, true>(m, lse, Dv, dk, dv, s, err, stream)
                      : launch_bwd_t<96, false, true>(m, lse, Dv, dk, dv, s, err, stream);
    return s.causal ? launch_bwd_t<96, true, false>(m, lse, Dv, dk, dv, s, err, stream)
                    : launch_bwd_t<96, false, false>(m, lse, Dv, dk, dv, s, err, stream);
  }
  if (with_dq)
    return s.causal ? launch_bwd_t<128, true, true>(m, lse, Dv, dk, dv, s, err, stream)
                    : launch_bwd_t<128, false, true>(m, lse, Dv, dk, dv, s, err, stream);
  return s.causal ? launch_bwd_t<128, true, false>(m, lse, Dv, dk, dv, s, err, stream)
                  : launch_bwd_t<128, false, false>(m, lse, Dv, dk, dv, s, err, stream);
}

}  // namespace fa
