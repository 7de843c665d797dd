/*
 * Exact attention oracle: a plain, slow, double-precision CPU statement of
 * what the attention path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the test suite, the smoke check and the CPU baseline
 * leg of the benchmark do.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (the plain definition; the tiled method reaches the same
 * result up to floating-point rounding order):
 *
 *   S = Q K^T * scale, with a causal mask of -inf on future keys
 *       ("FlashAttention: l'attenzione che non spreca memoria", the three
 *        steps S = QK^T/sqrt(d_k), P = softmax(S), O = PV of its opening
 *        section; "Flash Attention ... NVIDIA CUDA Tile", section
 *        "Atencion causal", mask 0 for i >= j and -inf for i < j)
 *   P = softmax(S) row by row, with the row maximum subtracted before exp
 *       (the stabilised one-shot softmax of "La online softmax, con i numeri")
 *   O = P V
 *   L = M + ln Z, the per-row log-sum-exp of the scaled, masked scores
 *       ("L'attention fusionnee", section "La passe arriere", L = m + ln(l))
 *
 * Backward, given dO ("L'attention fusionnee", section "La passe arriere"):
 *   dV = P^T dO
 *   dP = dO V^T
 *   dS = P o (dP - rowsum(P o dP))   -- the plain softmax Jacobian; the
 *                                       rowsum(dO o O) shortcut is NOT used
 *                                       here, it is checked against this.
 *   dQ = scale * dS K
 *   dK = scale * dS^T Q
 * Grouped-query attention: query head h reads key/value head h / G with
 * G = Hq / Hkv (contiguous groups, the QUERY_GROUP_SIZE parameter of the CUDA
 * Tile kernel signature).  The gradient of a shared key/value head is the sum
 * over the G query heads that read it (chain rule; the pages are silent).
 *
 * S and P are materialised in full for every head that is processed (or for
 * the requested rows only, see `rows`).  Nothing is tiled, fused or
 * reordered beyond plain loops over the definition.
 *
 * Layout: q, o, dq, do_: [B][Hq][Nq][d]; k, v, dk, dv: [B][Hkv][Nk][d];
 * lse and rowdot: [B][Hq][Nq] (or [B][Hq][n_rows] with `rows`); all row-major
 * doubles.  Query i sits at absolute position i + q_offset; under the causal
 * mask it sees keys j <= i + q_offset.  A query row that sees no key at all
 * (only possible with a negative offset) gets O = 0 and L = -inf.
 *
 * Return codes: 0 ok, 1 invalid argument, 2 out of host memory.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static int bad_shape(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 1 || d < 1) return 1;
  if (Hq % Hkv != 0) return 1;
  return 0;
}

/* One score row: s[j] = scale * <q_row, k_j>, or -inf where the causal mask
 * hides key j from absolute query position `pos`. */
static void score_row(const double* q_row, const double* k_head, int64_t Nk, int64_t d,
                      double scale, int causal, int64_t pos, double* s) {
  for (int64_t j = 0; j < Nk; ++j) {
    if (causal && j > pos) {
      s[j] = -INFINITY;
      continue;
    }
    const double* k_row = k_head + j * d;
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += q_row[c] * k_row[c];
    s[j] = scale * acc;
  }
}

/* Stabilised softmax of one row in place: s -> p.  Returns the row maximum M
 * and writes Z = sum_j exp(s_j - M).  A row of only -inf gives p = 0, Z = 0. */
static double softmax_row(double* s, int64_t Nk, double* Z_out) {
  double M = -INFINITY;
  for (int64_t j = 0; j < Nk; ++j)
    if (s[j] > M) M = s[j];
  if (M == -INFINITY) {
    for (int64_t j = 0; j < Nk; ++j) s[j] = 0.0;
    *Z_out = 0.0;
    return M;
  }
  double Z = 0.0;
  for (int64_t j = 0; j < Nk; ++j) {
    s[j] = exp(s[j] - M);
    Z += s[j];
  }
  for (int64_t j = 0; j < Nk; ++j) s[j] /= Z;
  *Z_out = Z;
  return M;
}

/*
 * Forward.  `rows` (may be NULL) selects which query rows of every head are
 * evaluated; then o is [B][Hq][n_rows][d] and lse [B][Hq][n_rows].
 * Per (b, hq) the n_rows x Nk matrices S and P are materialised.
 */
int oracle_attention_forward(const double* q, const double* k, const double* v, double* o,
                             double* lse, int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq,
                             int64_t Nk, int64_t d, double scale, int causal, int64_t q_offset,
                             const int64_t* rows, int64_t n_rows) {
  if (!q || !k || !v || !o || !lse) return 1;
  if (bad_shape(B, Hq, Hkv, Nq, Nk, d)) return 1;
  if (!rows) n_rows = Nq;
  if (n_rows < 0) return 1;
  if (rows)
    for (int64_t r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= Nq) return 1;
  const int64_t G = Hq / Hkv;
  const int64_t units = B * Hq;
  int status = 0;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t u = 0; u < units; ++u) {
    const int64_t b = u / Hq, h = u % Hq, hk = h / G;
    const double* q_head = q + (b * Hq + h) * Nq * d;
    const double* k_head = k + (b * Hkv + hk) * Nk * d;
    const double* v_head = v + (b * Hkv + hk) * Nk * d;
    double* o_head = o + (b * Hq + h) * n_rows * d;
    double* l_head = lse + (b * Hq + h) * n_rows;
    /* S, then P in its place: n_rows x Nk. */
    double* P = (double*)malloc((size_t)(n_rows > 0 ? n_rows : 1) * (size_t)Nk * sizeof(double));
    if (!P) {
#pragma omp atomic write
      status = 2;
      continue;
    }
    for (int64_t r = 0; r < n_rows; ++r) {
      const int64_t i = rows ? rows[r] : r;
      score_row(q_head + i * d, k_head, Nk, d, scale, causal, i + q_offset, P + r * Nk);
    }
    for (int64_t r = 0; r < n_rows; ++r) {
      double Z;
      const double M = softmax_row(P + r * Nk, Nk, &Z);
      l_head[r] = (M == -INFINITY) ? -INFINITY : M + log(Z);
    }
    for (int64_t r = 0; r < n_rows; ++r) {
      double* o_row = o_head + r * d;
      for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
      const double* p_row = P + r * Nk;
      for (int64_t j = 0; j < Nk; ++j) {
        const double p = p_row[j];
        if (p == 0.0) continue; /* masked or underflowed: contributes nothing */
        const double* v_row = v_head + j * d;
        for (int64_t c = 0; c < d; ++c) o_row[c] += p * v_row[c];
      }
    }
    free(P);
  }
  return status;
}

/*
 * Backward.  dq: [B][Hq][Nq][d]; dk, dv: [B][Hkv][Nk][d] (overwritten);
 * rowdot (may be NULL): [B][Hq][Nq], receives sum_j P_ij dP_ij, the quantity
 * the fused method replaces by rowsum(dO o O).
 * Parallel over (b, hkv) units so that the G heads of a group add into dk/dv
 * one after another.
 */
int oracle_attention_backward(const double* q, const double* k, const double* v,
                              const double* dout, double* dq, double* dk, double* dv,
                              double* rowdot, int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq,
                              int64_t Nk, int64_t d, double scale, int causal, int64_t q_offset) {
  if (!q || !k || !v || !dout || !dq || !dk || !dv) return 1;
  if (bad_shape(B, Hq, Hkv, Nq, Nk, d)) return 1;
  const int64_t G = Hq / Hkv;
  const int64_t units = B * Hkv;
  int status = 0;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t u = 0; u < units; ++u) {
    const int64_t b = u / Hkv, hk = u % Hkv;
    const double* k_head = k + (b * Hkv + hk) * Nk * d;
    const double* v_head = v + (b * Hkv + hk) * Nk * d;
    double* dk_head = dk + (b * Hkv + hk) * Nk * d;
    double* dv_head = dv + (b * Hkv + hk) * Nk * d;
    for (int64_t x = 0; x < Nk * d; ++x) {
      dk_head[x] = 0.0;
      dv_head[x] = 0.0;
    }
    const size_t mat = (size_t)(Nq > 0 ? Nq : 1) * (size_t)Nk;
    double* P = (double*)malloc(mat * sizeof(double));
    double* dP = (double*)malloc(mat * sizeof(double));
    if (!P || !dP) {
      free(P);
      free(dP);
#pragma omp atomic write
      status = 2;
      continue;
    }
    for (int64_t g = 0; g < G; ++g) {
      const int64_t h = hk * G + g;
      const double* q_head = q + (b * Hq + h) * Nq * d;
      const double* do_head = dout + (b * Hq + h) * Nq * d;
      double* dq_head = dq + (b * Hq + h) * Nq * d;
      /* P, materialised. */
      for (int64_t i = 0; i < Nq; ++i) {
        double Z;
        score_row(q_head + i * d, k_head, Nk, d, scale, causal, i + q_offset, P + i * Nk);
        softmax_row(P + i * Nk, Nk, &Z);
      }
      /* dP = dO V^T, materialised. */
      for (int64_t i = 0; i < Nq; ++i) {
        const double* do_row = do_head + i * d;
        for (int64_t j = 0; j < Nk; ++j) {
          const double* v_row = v_head + j * d;
          double acc = 0.0;
          for (int64_t c = 0; c < d; ++c) acc += do_row[c] * v_row[c];
          dP[i * Nk + j] = acc;
        }
      }
      /* dS = P o (dP - sum_k P_ik dP_ik), written over dP. */
      for (int64_t i = 0; i < Nq; ++i) {
        double r = 0.0;
        for (int64_t j = 0; j < Nk; ++j) r += P[i * Nk + j] * dP[i * Nk + j];
        if (rowdot) rowdot[(b * Hq + h) * Nq + i] = r;
        for (int64_t j = 0; j < Nk; ++j) dP[i * Nk + j] = P[i * Nk + j] * (dP[i * Nk + j] - r);
      }
      /* dV += P^T dO. */
      for (int64_t i = 0; i < Nq; ++i) {
        const double* do_row = do_head + i * d;
        for (int64_t j = 0; j < Nk; ++j) {
          const double p = P[i * Nk + j];
          if (p == 0.0) continue;
          double* dv_row = dv_head + j * d;
          for (int64_t c = 0; c < d; ++c) dv_row[c] += p * do_row[c];
        }
      }
      /* dQ = scale * dS K. */
      for (int64_t i = 0; i < Nq; ++i) {
        double* dq_row = dq_head + i * d;
        for (int64_t c = 0; c < d; ++c) dq_row[c] = 0.0;
        for (int64_t j = 0; j < Nk; ++j) {
          const double ds = dP[i * Nk + j];
          if (ds == 0.0) continue;
          const double* k_row = k_head + j * d;
          for (int64_t c = 0; c < d; ++c) dq_row[c] += ds * k_row[c];
        }
        for (int64_t c = 0; c < d; ++c) dq_row[c] *= scale;
      }
      /* dK += scale * dS^T Q. */
      for (int64_t i = 0; i < Nq; ++i) {
        const double* q_row = q_head + i * d;
        for (int64_t j = 0; j < Nk; ++j) {
          const double ds = dP[i * Nk + j];
          if (ds == 0.0) continue;
          double* dk_row = dk_head + j * d;
          for (int64_t c = 0; c < d; ++c) dk_row[c] += scale * ds * q_row[c];
        }
      }
    }
    free(P);
    free(dP);
  }
  return status;
}

/*
 * D[r] = sum_c a[r][c] * b[r][c] for `rows` rows of width d: the per-row
 * quantity the fused backward computes first ("L'attention fusionnee",
 * section "La passe arriere : recalculer plutot que garder": the sum of dP x P
 * over a row equals the sum of dO x O, one value per row).
 */
int oracle_row_dot(const double* a, const double* b, double* out, int64_t rows, int64_t d) {
  if (!a || !b || !out || rows < 0 || d < 1) return 1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += a[r * d + c] * b[r * d + c];
    out[r] = acc;
  }
  return 0;
}
