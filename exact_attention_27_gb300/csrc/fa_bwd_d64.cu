// Backward main kernel for head dimension 64 on sm_103a, pipelined.
//
// Same mathematics as the d = 128 kernel in fa_bwd.cu ("L'attention
// fusionnee", section "La passe arriere : recalculer plutot que garder": P
// rebuilt from L, dV = P^T dO, dS = P o (dP - D), dQ = dS K scale,
// dK = dS^T Q scale), arranged so that the tensor core and the threads work
// at the same time:
//
//  * One CTA owns 128 keys of one (batch, K/V head) and walks the query tiles
//    of every query head of the group in halves of 64 queries ("half-steps").
//  * K and V are copied once into tensor memory as bf16, so S^T = K Q^T and
//    dP^T = V dO^T take their A operand from TMEM; P^T and dS^T are written
//    back to TMEM as bf16, so dV += P^T dO and dK += dS^T Q do too.  Only
//    dQ = dS K reads both operands from shared memory (dS^T read MN-major).
//  * S^T/dP^T are double-buffered per half-step: while the threads turn half
//    h into P^T and dS^T, the tensor core finishes dV/dK of half h-1 and
//    computes S^T/dP^T of half h+1.  Both compute warpgroups work on every
//    half, each on 32 of its 64 query columns, which halves the dependent
//    chain each warp runs per half (the work there is latency-bound).
//  * A third warpgroup copies K and V into TMEM, stages L and D of upcoming
//    halves into a shared-memory ring and drains each query tile's dQ
//    through a swizzled staging tile and a TMA reduce-add into the fp32
//    accumulator.  At the end the two compute warpgroups write dK (times
//    scale) and dV, one each, while it drains the last dQ.
//  * The producer's lane initialises the barriers and issues the K, V and
//    first Q/dO loads before the CTA barrier, so that their latency overlaps
//    the tensor-memory allocation.
//
// Warps: 0-3 compute (query columns 0-31 of each half) and dK, 4-7 compute
// (columns 32-63) and dV, 8-11 L/D staging and dQ drain, 12 TMA producer,
// 13 MMA issuer.  448 threads, 1 CTA per SM.
//
// Tensor memory (512 columns):
//   [  0, 64) dK      [ 64,128) dV      [128,160) K bf16   [160,192) V bf16
//   [192,256) S^T buf0  [256,320) dP^T buf0  [320,384) S^T buf1  [384,448) dP^T buf1
//   [448,512) dQ of the current query tile
// Warpgroup w writes its P^T (bf16, 16 columns) at columns [32w, 32w+16) of
// the S^T buffer, over S^T columns it has itself just read, and its dS^T the
// same way in the dP^T buffer; the MMAs address the two 16-column pieces.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct Cfg64 {
  static constexpr int BK = 128;                 // keys per CTA
  static constexpr int BQ = 128;                 // queries per tile (two halves)
  static constexpr int TILE = 128 * 128;         // 128 rows x 64 bf16
  static constexpr int NSQ = 3;                  // Q / dO stages
  // V is only needed until it has been copied into tensor memory; its
  // region then holds the first box of the dQ staging tile.
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_STG = OFF_V;                  // dQ staging: 2 boxes 128 x 32 fp32
  static constexpr int OFF_Q = OFF_STG + 2 * TILE;
  static constexpr int OFF_DO = OFF_Q + NSQ * TILE;
  static constexpr int OFF_DS = OFF_DO + NSQ * TILE;  // 2 x (128 keys x 128 queries bf16)
  static constexpr int DS_BYTES = 2 * TILE;
  // L/D ring: NLD slots of one half-step each, -L*log2e[64] then -D[64]
  static constexpr int NLD = 6;
  static constexpr int OFF_LD = OFF_DS + 2 * DS_BYTES;
  static constexpr int OFF_BAR = OFF_LD + NLD * 128 * 4;
  // barriers
  static constexpr int B_KV = 0;
  static constexpr int B_KVT = 1;                 // K, V copied into TMEM (4 warp arrivals)
  static constexpr int B_QDFULL = 2;              // [NSQ]
  static constexpr int B_QDEMPTY = B_QDFULL + NSQ;
  static constexpr int B_SDP = B_QDEMPTY + NSQ;   // [2] S^T/dP^T of a half ready
  static constexpr int B_PDS = B_SDP + 2;         // [2] P^T/dS^T of a half ready (8 warp arrivals)
  static constexpr int B_DQFULL = B_PDS + 2;      // dQ of a tile in TMEM
  static constexpr int B_DQFREE = B_DQFULL + 1;   // dQ drained (4 warp arrivals)
  static constexpr int B_WG = B_DQFREE + 1;       // drain-warpgroup internal sync (4 warp arrivals)
  static constexpr int B_LDFULL = B_WG + 1;       // [NLD] L/D slot filled (4 warp arrivals)
  static constexpr int B_LDEMPTY = B_LDFULL + NLD; // [NLD] L/D slot read (8 warp arrivals)
  static constexpr int B_FINAL = B_LDEMPTY + NLD;  // every MMA issued has completed (once)
  static constexpr int B_DRAIN = B_FINAL + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + 8 * NBAR;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int THREADS = 448;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_DK = 0, COL_DV = 64, COL_KT = 128, COL_VT = 160;
  static constexpr uint32_t COL_BUF = 192;        // + 128 * buf: S^T, + 64: dP^T
  static constexpr uint32_t COL_DQ = 448;
};

struct Params64 {
  const float* lse;
  const float* Dvec;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int N, Hq, Hkv, G, n_qtiles;
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

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// DQ = false builds the dK/dV-only kernel of the deterministic backward: no
// dQ product, no dQ drain and no dS^T in shared memory; the per-tile
// completion barrier still paces the L/D ring.
template <bool CAUSAL, bool DQ>
__global__ void __launch_bounds__(448, 1)
    fa_bwd64_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmdQ, const Params64 p) {
  using C = Cfg64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int wg = warp >> 2;  // 0, 1 compute; 2 drain; 3 = warps 12, 13
  const int n_kv_units = gridDim.x / ((p.N + C::BK - 1) / C::BK);
  // Heaviest key tiles (most query tiles under the causal mask) first.
  const int jt = static_cast<int>(blockIdx.x) / n_kv_units;
  const int kvz = static_cast<int>(blockIdx.x) - jt * n_kv_units;  // flattened (batch, kv head)
  const int b = kvz / p.Hkv;
  const int hkv = kvz - b * p.Hkv;
  const int i0 = CAUSAL ? jt : 0;
  const int per_head = p.n_qtiles - i0;
  const int n_steps = p.G * per_head;
  const int n_half = 2 * n_steps;

  const uint32_t sK = sbase + C::OFF_K;
  const uint32_t sV = sbase + C::OFF_V;
  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t sdO = sbase + C::OFF_DO;
  const uint32_t sDS = sbase + C::OFF_DS;
  const uint32_t sSTG = sbase + C::OFF_STG;

  // step -> (query head within the group, query tile)
  auto step_coords = [&](int s, int& bhq, int& it) {
    const int g = s / per_head;
    it = i0 + (s - g * per_head);
    bhq = b * p.Hq + hkv * p.G + g;
  };

  // The producer's lane initialises the barriers and issues the loads of K,
  // V and the first Q/dO stages at once, so that their latency overlaps the
  // tensor-memory allocation and the CTA barrier below.  (K, V, Q and dO are
  // inputs of the backward, which this grid may read before it waits for
  // the grid before it.)
  const int first_loads = min(C::NSQ, n_steps);
  if (warp == 12 && elect_one()) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    mbar_init(bar(C::B_KV), 1);
    mbar_init(bar(C::B_KVT), 4);  // one arrival per warp of the drain warpgroup
    for (int s = 0; s < C::NSQ; ++s) {
      mbar_init(bar(C::B_QDFULL + s), 1);
      mbar_init(bar(C::B_QDEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_SDP + s), 1);
      mbar_init(bar(C::B_PDS + s), 8);  // both compute warpgroups
    }
    mbar_init(bar(C::B_DQFULL), 1);
    mbar_init(bar(C::B_DQFREE), 4);
    mbar_init(bar(C::B_WG), 4);
    for (int s = 0; s < C::NLD; ++s) {
      mbar_init(bar(C::B_LDFULL + s), 4);
      mbar_init(bar(C::B_LDEMPTY + s), 8);
    }
    mbar_init(bar(C::B_FINAL), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_barrier_init();
    mbar_arrive_expect_tx(bar(C::B_KV), 2 * C::TILE);
    tma_load_3d(sK, &tmK, bar(C::B_KV), 0, jt * C::BK, kvz);
    tma_load_3d(sV, &tmV, bar(C::B_KV), 0, jt * C::BK, kvz);
    for (int s = 0; s < first_loads; ++s) {
      int bhq, it;
      step_coords(s, bhq, it);
      mbar_arrive_expect_tx(bar(C::B_QDFULL + s), 2 * C::TILE);
      tma_load_3d(sQ + s * C::TILE, &tmQ, bar(C::B_QDFULL + s), 0, it * C::BQ, bhq);
      tma_load_3d(sdO + s * C::TILE, &tmdO, bar(C::B_QDFULL + s), 0, it * C::BQ, bhq);
    }
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      // K, V and steps 0 .. first_loads - 1 were issued before the CTA barrier.
      int issued = first_loads;
      for (int s = first_loads; s < n_steps; ++s) {
        const int st = s % C::NSQ;
        if (s >= C::NSQ && !mbar_wait(bar(C::B_QDEMPTY + st), ((s / C::NSQ) - 1) & 1,
                                      abort_flag, p.err, kErrTimeoutLoad))
          break;
        int bhq, it;
        step_coords(s, bhq, it);
        mbar_arrive_expect_tx(bar(C::B_QDFULL + st), 2 * C::TILE);
        tma_load_3d(sQ + st * C::TILE, &tmQ, bar(C::B_QDFULL + st), 0, it * C::BQ, bhq);
        tma_load_3d(sdO + st * C::TILE, &tmdO, bar(C::B_QDFULL + st), 0, it * C::BQ, bhq);
        issued = s + 1;
      }
      if (*abort_flag) {
        mbar_wait_timed(bar(C::B_KV), 0);
        for (int s2 = max(0, issued - C::NSQ); s2 < issued; ++s2)
          mbar_wait_timed(bar(C::B_QDFULL + s2 % C::NSQ), (s2 / C::NSQ) & 1);
      }
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t ID_SDP = idesc_bf16_f32(128, 64, false, false);  // S^T, dP^T
      constexpr uint32_t ID_KV = idesc_bf16_f32(128, 64, false, true);    // dV, dK
      constexpr uint32_t ID_Q = idesc_bf16_f32(128, 64, true, true);      // dQ
      // Descriptors built once; k-steps move them by compile-time offsets.
      const uint64_t q_kmaj = smem_desc_sw128(sQ, 16, 1024);        // Q as K-major B
      const uint64_t do_kmaj = smem_desc_sw128(sdO, 16, 1024);
      const uint64_t q_mn = smem_desc_sw128(sQ, C::TILE, 1024);     // Q as MN-major B
      const uint64_t do_mn = smem_desc_sw128(sdO, C::TILE, 1024);
      const uint64_t ds_mn = smem_desc_sw128(sDS, C::TILE, 1024);   // dS (query rows) as A
      const uint64_t k_mn = smem_desc_sw128(sK, C::TILE, 1024);     // K as MN-major B
      bool ok = mbar_wait(bar(C::B_KVT), 0, abort_flag, p.err, kErrTimeoutMma);
      // S^T and dP^T of half h into buffer h & 1.
      auto issue_sdp = [&](int h) -> bool {
        const int s = h >> 1, a = h & 1, st = s % C::NSQ;
        if (a == 0 && !mbar_wait(bar(C::B_QDFULL + st), (s / C::NSQ) & 1, abort_flag, p.err,
                                 kErrTimeoutMma))
          return false;
        tc_fence_after();
        const uint32_t buf = tmem + C::COL_BUF + 128 * (h & 1);
        const uint32_t off = st * C::TILE + a * 8192;
        const uint64_t qd = desc_add(q_kmaj, off), dd = desc_add(do_kmaj, off);
        mma_ts_k<ID_SDP, 0>(buf, tmem + C::COL_KT, qd);
        mma_ts_k<ID_SDP, 1>(buf, tmem + C::COL_KT + 8, desc_add(qd, 32));
        mma_ts_k<ID_SDP, 1>(buf, tmem + C::COL_KT + 16, desc_add(qd, 64));
        mma_ts_k<ID_SDP, 1>(buf, tmem + C::COL_KT + 24, desc_add(qd, 96));
        mma_ts_k<ID_SDP, 0>(buf + 64, tmem + C::COL_VT, dd);
        mma_ts_k<ID_SDP, 1>(buf + 64, tmem + C::COL_VT + 8, desc_add(dd, 32));
        mma_ts_k<ID_SDP, 1>(buf + 64, tmem + C::COL_VT + 16, desc_add(dd, 64));
        mma_ts_k<ID_SDP, 1>(buf + 64, tmem + C::COL_VT + 24, desc_add(dd, 96));
        mma_commit(bar(C::B_SDP + (h & 1)));
        return true;
      };
      if (ok) ok = issue_sdp(0);
      if (ok && n_half > 1) ok = issue_sdp(1);
      for (int h = 0; ok && h < n_half; ++h) {
        const int s = h >> 1, a = h & 1, st = s % C::NSQ;
        if (!mbar_wait(bar(C::B_PDS + a), (h >> 1) & 1, abort_flag, p.err, kErrTimeoutMma)) break;
        tc_fence_after();
        const uint32_t buf = tmem + C::COL_BUF + 128 * a;
        const uint32_t off = st * C::TILE + a * 8192;
        const uint64_t qd = desc_add(q_mn, off), dd = desc_add(do_mn, off);
        // dV += P^T dO_h ; dK += dS^T Q_h  (64 queries = 4 steps of 16)
        // P^T / dS^T of queries 16kk.. sit at columns (kk/2)*32 + (kk%2)*8.
        if (h == 0) {
          mma_ts_k<ID_KV, 0>(tmem + C::COL_DV, buf, dd);
          mma_ts_k<ID_KV, 0>(tmem + C::COL_DK, buf + 64, qd);
        } else {
          mma_ts_k<ID_KV, 1>(tmem + C::COL_DV, buf, dd);
          mma_ts_k<ID_KV, 1>(tmem + C::COL_DK, buf + 64, qd);
        }
#pragma unroll
        for (int kk = 1; kk < 4; ++kk) {
          const uint32_t col = (kk >> 1) * 32 + (kk & 1) * 8;
          mma_ts_k<ID_KV, 1>(tmem + C::COL_DV, buf + col, desc_add(dd, kk * 2048));
          mma_ts_k<ID_KV, 1>(tmem + C::COL_DK, buf + 64 + col, desc_add(qd, kk * 2048));
        }
        // Q_h and dO_h of the tile are not read after the second half's dV/dK.
        if (a == 1) mma_commit(bar(C::B_QDEMPTY + st));
        // Queue the next S^T/dP^T before possibly waiting for the dQ drain, so
        // that the tensor core keeps working meanwhile.
        if (h + 2 < n_half && !issue_sdp(h + 2)) break;
        if (a == 1 && DQ) {
          if (s > 0) {
            if (!mbar_wait(bar(C::B_DQFREE), (s - 1) & 1, abort_flag, p.err, kErrTimeoutMma))
              break;
            tc_fence_after();
          }
          // dQ = dS K_j: A = dS (query rows) read MN-major from the dS^T tile.
          const uint64_t dsd = desc_add(ds_mn, (s & 1) * C::DS_BYTES);
          mma_ss_k<ID_Q, 0>(tmem + C::COL_DQ, dsd, k_mn);
#pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            mma_ss_k<ID_Q, 1>(tmem + C::COL_DQ, desc_add(dsd, kk * 2048), desc_add(k_mn, kk * 2048));
          mma_commit(bar(C::B_DQFULL));
        }
        // Once, after the last half: everything issued has completed.  (A
        // barrier that completes once per tile could not tell its last phase
        // apart from an earlier one by parity when nothing holds it back.)
        if (h == n_half - 1) mma_commit(bar(C::B_FINAL));
      }
      if (*abort_flag) {
        mma_commit(bar(C::B_DRAIN));
        mbar_wait_timed(bar(C::B_DRAIN), 0);
      }
    }
  } else if (wg < 2) {
    // ------------------------------------------------------------ compute (key rows)
    // Warpgroup wg handles query columns [32 wg, 32 wg + 32) of every half.
    const int t = threadIdx.x & 127;  // key row
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int key = jt * C::BK + t;
    const bool key_live = key < p.N;
    const float c = p.scale_log2;
    bool ok = true;
    for (int h = 0; h < n_half; ++h) {
      const int s = h >> 1, a = h & 1;
      int bhq, it;
      step_coords(s, bhq, it);
      const int q0 = it * C::BQ + a * 64 + wg * 32;  // first query of this warpgroup's columns
      // S^T/dP^T of this half.  Its completion also means that the dQ product
      // of tile s - 2 has read the dS^T buffer this tile writes again: that
      // product was issued, by the same thread, before this half's S^T/dP^T,
      // and a commit tracks every earlier tcgen05 operation of its thread.
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SDP + a), (h >> 1) & 1, abort_flag, p.err,
                                             kErrTimeoutSoftmax));
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_LDFULL + h % C::NLD), (h / C::NLD) & 1,
                                             abort_flag, p.err, kErrTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      const uint32_t sbuf = tmem + lane_off + C::COL_BUF + 128 * a + 32 * wg;
      const float* slot = reinterpret_cast<const float*>(smem + C::OFF_LD) + (h % C::NLD) * 128;
      const float4* L4 = reinterpret_cast<const float4*>(slot + 32 * wg);       // -L log2e
      const float4* D4 = reinterpret_cast<const float4*>(slot + 64 + 32 * wg);  // -D
      uint32_t sv[32], dpv[32];
      tmem_ld32(sbuf, sv);
      tmem_ld32(sbuf + 64, dpv);
      // Masking is needed only on the diagonal tile and for keys past N;
      // warp-uniform, so the common case runs without per-element tests.
      const bool masked = __any_sync(0xffffffffu, (CAUSAL && it == jt) || !key_live);
      tmem_wait_ld();
      uint32_t pk[16], dk16[16];
      const uint64_t c2 = f2_pack(c, c);
#pragma unroll
      for (int u4 = 0; u4 < 8; ++u4) {
        const float4 nl = L4[u4];
        const float4 nd = D4[u4];
        float pv[4];
        // exp2 argument s c - L log2e on pairs
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[4 * u4]), __uint_as_float(sv[4 * u4 + 1])),
                         c2, f2_pack(nl.x, nl.y)),
                  pv[0], pv[1]);
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[4 * u4 + 2]), __uint_as_float(sv[4 * u4 + 3])),
                         c2, f2_pack(nl.z, nl.w)),
                  pv[2], pv[3]);
#pragma unroll
        for (int e = 0; e < 4; ++e) pv[e] = ex2_approx(pv[e]);
        if (masked) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (!key_live || (CAUSAL && key > q0 + u4 * 4 + e)) pv[e] = 0.0f;
        }
        // dS = P o (dP - D) on pairs
        const uint64_t ds01 = f2_mul(
            f2_pack(pv[0], pv[1]),
            f2_add(f2_pack(__uint_as_float(dpv[4 * u4]), __uint_as_float(dpv[4 * u4 + 1])),
                   f2_pack(nd.x, nd.y)));
        const uint64_t ds23 = f2_mul(
            f2_pack(pv[2], pv[3]),
            f2_add(f2_pack(__uint_as_float(dpv[4 * u4 + 2]), __uint_as_float(dpv[4 * u4 + 3])),
                   f2_pack(nd.z, nd.w)));
        float dsv[4];
        f2_unpack(ds01, dsv[0], dsv[1]);
        f2_unpack(ds23, dsv[2], dsv[3]);
        pk[2 * u4] = pack_bf16x2(pv[0], pv[1]);
        pk[2 * u4 + 1] = pack_bf16x2(pv[2], pv[3]);
        dk16[2 * u4] = pack_bf16x2(dsv[0], dsv[1]);
        dk16[2 * u4 + 1] = pack_bf16x2(dsv[2], dsv[3]);
      }
      tmem_st16(sbuf, pk);         // P^T over this warpgroup's S^T columns
      tmem_st16(sbuf + 64, dk16);  // dS^T over its dP^T columns
      if (DQ) {
        // dS^T row t, queries 32wg .. 32wg+31 of the half: chunks 4wg..4wg+3 of block a.
        const uint32_t ds_blk = sDS + (s & 1) * C::DS_BYTES + a * C::TILE;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          st_shared_v4(ds_blk + sw128(t, wg * 4 + q4), dk16[4 * q4], dk16[4 * q4 + 1],
                       dk16[4 * q4 + 2], dk16[4 * q4 + 3]);
      }
      tmem_wait_st();
      if (DQ) fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive_warp(bar(C::B_PDS + a));
      mbar_arrive_warp(bar(C::B_LDEMPTY + h % C::NLD));  // this half's L/D are no longer read
    }
    // ---- epilogue, once every MMA has completed: warpgroup 0 writes dK
    // (times scale), warpgroup 1 dV, while the drain finishes the last dQ.
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_FINAL), 0, abort_flag, p.err,
                                                   kErrTimeoutEpilogue));
    if (ok) {
      tc_fence_after();
      const float mul = wg == 0 ? p.scale : 1.0f;
      __nv_bfloat16* row = (wg == 0 ? p.dk : p.dv) +
                           (static_cast<size_t>(kvz) * p.N + (key_live ? key : 0)) * 64;
#pragma unroll
      for (int q4 = 0; q4 < 2; ++q4) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + (wg == 0 ? C::COL_DK : C::COL_DV) + q4 * 32, r);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          pk[u] = pack_bf16x2(__uint_as_float(r[2 * u]) * mul, __uint_as_float(r[2 * u + 1]) * mul);
        if (key_live) {
          uint4* dst = reinterpret_cast<uint4*>(row + q4 * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dst[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
    }
  } else if (wg == 2) {
    // ------------------------------------------------------------ K/V -> TMEM, L/D ring, dQ drain
    const int t = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t wg_phase = 0;
    bool ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_KV), 0, abort_flag, p.err,
                                                kErrTimeoutOther));
    if (ok) {
      // Row t of K and V (64 bf16 = 8 swizzled 16-byte chunks) -> 32 TMEM columns.
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t src = which == 0 ? sK : sV;
        uint32_t r[32];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 v = ld_shared_v4(src + sw128(t, ch));
          r[4 * ch] = v.x;
          r[4 * ch + 1] = v.y;
          r[4 * ch + 2] = v.z;
          r[4 * ch + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + (which == 0 ? C::COL_KT : C::COL_VT), r);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(bar(C::B_KVT));
    }
    auto wg_sync = [&]() -> bool {
      mbar_arrive_warp(bar(C::B_WG));
      const bool r = mbar_wait(bar(C::B_WG), wg_phase & 1, abort_flag, p.err, kErrTimeoutOther);
      ++wg_phase;
      return __all_sync(0xffffffffu, r);
    };
    // L and D of half h: thread t < 64 loads L of query t of the half, t >= 64
    // D of query t - 64.  Rows past N read as L = +inf (so P = 0) and D = -0.
    // The raw value is kept until it is stored, so that nothing waits for the
    // load before then: the loads for tile s + 3 are in flight while tile s's
    // dQ is drained.
    auto load_ld = [&](int h) -> float {
      if (h >= n_half) return 0.0f;
      int bhq, it;
      step_coords(h >> 1, bhq, it);
      const int qrow = it * C::BQ + (h & 1) * 64 + (t & 63);
      if (qrow >= p.N) return t < 64 ? INFINITY : -0.0f;
      const size_t idx = static_cast<size_t>(bhq) * p.N + qrow;
      return t < 64 ? p.lse[idx] : p.Dvec[idx];
    };
    // Ring slot h % NLD takes -L log2e and -D (negated, so the compute warps add them).
    auto store_ld = [&](int h, float raw) {
      if (h >= n_half) return;
      reinterpret_cast<float*>(smem + C::OFF_LD)[(h % C::NLD) * 128 + t] =
          t < 64 ? -raw * kLog2e : -raw;
      mbar_arrive_warp(bar(C::B_LDFULL + h % C::NLD));
    };
    // This warpgroup alone reads what the row-dot pass (the grid before this
    // one) writes: D, and the zeroed dQ accumulator the reduces add into.
    // Everything before this point (and the other roles' K, V, Q and dO
    // loads and first products) may run while that grid drains.
    grid_dependency_wait();
    // Halves of tiles 0..2 first; then, once the compute warps have read the
    // slots of tile s, the halves of tile s + 3 go into them.  The loads for
    // tile s + 3 are issued before waiting for tile s.
    for (int h = 0; h < C::NLD; ++h) store_ld(h, load_ld(h));
    for (int s = 0; ok && s < n_steps; ++s) {
      int bhq, it;
      step_coords(s, bhq, it);
      const float ld_next0 = load_ld(2 * (s + 3));
      const float ld_next1 = load_ld(2 * (s + 3) + 1);
      if (DQ) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::B_DQFULL), s & 1, abort_flag, p.err, kErrTimeoutOther));
      if (!ok) break;
      tc_fence_after();
      uint32_t a[32], bb[32];
      tmem_ld32(tmem + lane_off + C::COL_DQ, a);
      tmem_ld32(tmem + lane_off + C::COL_DQ + 32, bb);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(bar(C::B_DQFREE));  // dQ columns may be overwritten now
      if (t == 0) bulk_wait_group_read0();  // staging free again
      if (!(ok = wg_sync())) break;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        st_shared_v4(sSTG + sw128(t, ch), a[4 * ch], a[4 * ch + 1], a[4 * ch + 2], a[4 * ch + 3]);
        st_shared_v4(sSTG + C::TILE + sw128(t, ch), bb[4 * ch], bb[4 * ch + 1], bb[4 * ch + 2],
                     bb[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      if (!(ok = wg_sync())) break;
      if (t == 0) {
        tma_reduce_add_3d(&tmdQ, sSTG, 0, it * C::BQ, bhq);
        tma_reduce_add_3d(&tmdQ, sSTG + C::TILE, 32, it * C::BQ, bhq);
        bulk_commit_group();
      }
      }  // DQ
      // The ring slots of tile s take tile s + 3 once both halves of tile s
      // were read (a barrier per slot, so that the refills cannot run ahead).
      for (int x = 0; x < 2 && 2 * (s + 3) + x < n_half; ++x) {
        const int h = 2 * s + x;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_LDEMPTY + h % C::NLD), (h / C::NLD) & 1,
                                               abort_flag, p.err, kErrTimeoutOther));
        if (!ok) break;
        store_ld(2 * (s + 3) + x, x == 0 ? ld_next0 : ld_next1);
      }
      if (!ok) break;
    }
    // Only the staging tile's reads must be over before the CTA's shared
    // memory is released; the reduces' writes complete on their own, and the
    // dQ finalisation reads the accumulator only after this grid has completed.
    if (t == 0) bulk_wait_group_read0();
    __syncwarp();
    grid_launch_dependents();  // the dQ finalisation may be scheduled
  }

  // Every warp reconverges first: in the TMA and MMA warps only one lane did
  // the work, and the CTA barrier below must count whole, converged warps.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <bool CAUSAL, bool DQ>
cudaError_t launch_t(const BwdMaps& m, const float* lse, const float* Dv, void* dk, void* dv,
                     const AttnShape& s, uint32_t* err, cudaStream_t stream) {
  using C = Cfg64;
  auto kern = fa_bwd64_kernel<CAUSAL, DQ>;
  cudaError_t e = set_smem_limit_once<fa_bwd64_kernel<CAUSAL, DQ>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  Params64 p;
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
  const long long n_ktiles = (s.N + C::BK - 1) / C::BK;
  const long long grid = n_ktiles * s.B * s.Hkv;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_dependent(kern, dim3(static_cast<unsigned>(grid)), dim3(C::THREADS),
                          C::SMEM_BYTES, stream, m.q, m.k, m.v, m.dO, m.dq_acc, p);
}

}  // namespace

cudaError_t launch_backward_d64(const BwdMaps& m, const float* lse, const float* Dv, void* dk,
                                void* dv, const AttnShape& s, uint32_t* err, cudaStream_t stream,
                                bool with_dq) {
  if (with_dq)
    return s.causal ? launch_t<true, true>(m, lse, Dv, dk, dv, s, err, stream)
                    : launch_t<false, true>(m, lse, Dv, dk, dv, s, err, stream);
  return s.causal ? launch_t<true, false>(m, lse, Dv, dk, dv, s, err, stream)
                  : launch_t<false, false>(m, lse, Dv, dk, dv, s, err, stream);
}

}  // namespace fa
