/*
 * Plain CPU oracle for exact softmax attention (test infrastructure only).
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load this library.  The product path never calls it and shares no
 * code with it.
 *
 * What it computes, per (batch b, head h), with every 16-bit input widened
 * exactly to double first:
 *
 *   s_ij = scale * sum_k q_ik k_jk        "Standard Attention": S = QK^T
 *                                         (Flash Attention 2 page, Standard
 *                                         Attention; the scale 1/sqrt(d) is the
 *                                         one of FlashAttention V2 in depth
 *                                         section 6.1 and of Lesson 6.6
 *                                         "A quick recap of standard attention")
 *   causal: key j is visible to query i only when j <= i
 *                                         (Flash Attention 2 page, Causal
 *                                         masking, the mask M; FlashAttention
 *                                         V2 in depth section 5.1)
 *   m_i  = max over visible j of s_ij
 *   p_ij = exp(s_ij - m_i) / sum_j exp(s_ij - m_i)     row softmax
 *   o_i  = sum_j p_ij v_j                              O = PV
 *   L_i  = m_i + ln sum_j exp(s_ij - m_i)              the logsumexp that
 *                                         FlashAttention V2 in depth sections
 *                                         6.1 and 7.1 store for the backward
 *
 * It is the plain definition: one full row of S is formed, then the full row
 * of P, then the row of O.  There is no tiling, no online softmax and no
 * reordering beyond the row-by-row evaluation; masked keys (exp(-inf) = 0)
 * are left out of the sums, which adds nothing to them.
 *
 * Parity: pinned by the tests against the worked example of the Flash
 * Attention 2 page, the one-row practice of Lesson 6.6, closed forms and
 * invariants (row sums, identical keys, single key, constant values, causal
 * row 0) and a high-precision brute force on tiny inputs.
 *
 * Backward (the gradients of the forward pass for an upstream gradient dO,
 * FlashAttention V2 in depth section 7 and Lesson 6.6 "Recomputation in the
 * backward pass"), per (b, h), by the definition of the softmax Jacobian:
 *
 *   P   = softmax_row(S) as above (visible keys only)
 *   dV  = P^T dO
 *   dP  = dO V^T
 *   D_i = sum_j P_ij dP_ij          (section 7.3 shows it equals rowsum(dO o O))
 *   dS  = P o (dP - D)              (o: elementwise)
 *   dQ  = scale dS K,   dK = scale dS^T Q
 *
 * Rows are done first (P row, dP row, D_i, dQ_i), then keys (dK_j, dV_j
 * summed over the rows that see key j, with P_ij and dS_ij rebuilt from the
 * row statistics of the first pass).  Pinned by central finite differences
 * of the forward definition, the identity of section 7.3 and invariants.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_FP16 = 0, ORACLE_BF16 = 1 };
enum { ORACLE_OK = 0, ORACLE_ERR_ARG = 1, ORACLE_ERR_NOMEM = 2 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -24);               /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        mag = f ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16: the upper 16 bits of an IEEE 754 binary32
 * (1 sign bit, 8 exponent bits with bias 127, 7 fraction bits). */
static double bfloat_bits_to_double(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -133);              /* f * 2^-126 * 2^-7 */
    } else if (e == 255) {
        mag = f ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(128 + f), e - 134);   /* (1 + f/128) * 2^(e-127) */
    }
    return sign ? -mag : mag;
}

static double widen(uint16_t bits, int dtype) {
    return dtype == ORACLE_BF16 ? bfloat_bits_to_double(bits) : half_bits_to_double(bits);
}

/* Exact widening of n 16-bit values, exported so tests can check it against a
 * library conversion. */
int oracle_widen(const uint16_t* src, int dtype, int64_t n, double* dst) {
    if (!src || !dst || n < 0 || (dtype != ORACLE_FP16 && dtype != ORACLE_BF16)) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) dst[i] = widen(src[i], dtype);
    return ORACLE_OK;
}

/* One query row i of one (b, h) slice, by the definition above.
 * qrow: d doubles; kmat, vmat: N x d doubles (row-major); srow: N doubles of
 * scratch for the materialised S row (then P row). */
static void attention_row(const double* qrow, const double* kmat, const double* vmat,
                          int64_t N, int64_t d, double scale, int causal, int64_t i,
                          double* srow, double* orow, double* lse) {
    int64_t nvis = causal ? (i + 1 < N ? i + 1 : N) : N;
    /* S row: s_ij = scale * q_i . k_j */
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        const double* kj = kmat + j * d;
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c) acc += qrow[c] * kj[c];
        srow[j] = scale * acc;
        if (srow[j] > m) m = srow[j];
    }
    /* P row: exp(s - m) / sum */
    double sum = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        srow[j] = exp(srow[j] - m);
        sum += srow[j];
    }
    for (int64_t j = 0; j < nvis; ++j) srow[j] /= sum;
    /* O row: sum_j p_ij v_j */
    for (int64_t c = 0; c < d; ++c) orow[c] = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        const double* vj = vmat + j * d;
        double p = srow[j];
        for (int64_t c = 0; c < d; ++c) orow[c] += p * vj[c];
    }
    *lse = m + log(sum);
}

static int check_args(const void* q, const void* k, const void* v, int dtype, int64_t B, int64_t H,
                      int64_t N, int64_t d, double scale) {
    if (!q || !k || !v) return ORACLE_ERR_ARG;
    if (dtype != ORACLE_FP16 && dtype != ORACLE_BF16) return ORACLE_ERR_ARG;
    if (B < 1 || H < 1 || N < 1 || d < 1) return ORACLE_ERR_ARG;
    if (!isfinite(scale)) return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/*
 * Selected rows.  q, k, v: [B, H, N, d] 16-bit bit patterns (dtype 0 = fp16,
 * 1 = bf16).  For each sample t, bh_idx[t] in [0, B*H) names the (b, h) slice
 * (bh = b*H + h) and row_idx[t] in [0, N) the query row; o_out receives
 * count x d doubles, lse_out count doubles (natural log).  Samples of the same
 * slice should be adjacent so that slice's K and V are widened once.
 * threads <= 0 uses the OpenMP default.
 */
int oracle_attention_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype,
                          int64_t B, int64_t H, int64_t N, int64_t d, double scale, int causal,
                          const int64_t* bh_idx, const int64_t* row_idx, int64_t count,
                          double* o_out, double* lse_out, int threads) {
    int rc = check_args(q, k, v, dtype, B, H, N, d, scale);
    if (rc) return rc;
    if (count < 0 || (count > 0 && (!bh_idx || !row_idx || !o_out || !lse_out))) return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < count; ++t)
        if (bh_idx[t] < 0 || bh_idx[t] >= B * H || row_idx[t] < 0 || row_idx[t] >= N) return ORACLE_ERR_ARG;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
    double* kmat = (double*)malloc(sizeof(double) * (size_t)(N * d));
    double* vmat = (double*)malloc(sizeof(double) * (size_t)(N * d));
    if (!kmat || !vmat) { free(kmat); free(vmat); return ORACLE_ERR_NOMEM; }
    int status = ORACLE_OK;
    int64_t t0 = 0;
    while (t0 < count) {
        int64_t bh = bh_idx[t0];
        int64_t t1 = t0;
        while (t1 < count && bh_idx[t1] == bh) ++t1;
        const uint16_t* ks = k + bh * N * d;
        const uint16_t* vs = v + bh * N * d;
        for (int64_t x = 0; x < N * d; ++x) { kmat[x] = widen(ks[x], dtype); vmat[x] = widen(vs[x], dtype); }
        int nomem = 0;
#pragma omp parallel reduction(| : nomem)
        {
            double* srow = (double*)malloc(sizeof(double) * (size_t)N);
            double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
            if (!srow || !qrow) {
                nomem = 1;
            } else {
#pragma omp for schedule(dynamic, 1)
                for (int64_t t = t0; t < t1; ++t) {
                    int64_t i = row_idx[t];
                    const uint16_t* qs = q + (bh * N + i) * d;
                    for (int64_t c = 0; c < d; ++c) qrow[c] = widen(qs[c], dtype);
                    attention_row(qrow, kmat, vmat, N, d, scale, causal, i, srow, o_out + t * d, lse_out + t);
                }
            }
            free(srow);
            free(qrow);
        }
        if (nomem) { status = ORACLE_ERR_NOMEM; break; }
        t0 = t1;
    }
    free(kmat);
    free(vmat);
    return status;
}

/* Every row: o_out [B, H, N, d] doubles, lse_out [B, H, N] doubles. */
int oracle_attention_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype,
                         int64_t B, int64_t H, int64_t N, int64_t d, double scale, int causal,
                         double* o_out, double* lse_out, int threads) {
    int rc = check_args(q, k, v, dtype, B, H, N, d, scale);
    if (rc) return rc;
    if (!o_out || !lse_out) return ORACLE_ERR_ARG;
    int64_t* bh_idx = (int64_t*)malloc(sizeof(int64_t) * (size_t)N);
    int64_t* row_idx = (int64_t*)malloc(sizeof(int64_t) * (size_t)N);
    if (!bh_idx || !row_idx) { free(bh_idx); free(row_idx); return ORACLE_ERR_NOMEM; }
    for (int64_t bh = 0; bh < B * H && rc == ORACLE_OK; ++bh) {
        for (int64_t i = 0; i < N; ++i) { bh_idx[i] = bh; row_idx[i] = i; }
        rc = oracle_attention_rows(q, k, v, dtype, B, H, N, d, scale, causal, bh_idx, row_idx, N,
                                   o_out + bh * N * d, lse_out + bh * N, threads);
    }
    free(bh_idx);
    free(row_idx);
    return rc;
}

/* ------------------------------------------------------------------ fp64 inputs */

static int check_args_f64(const double* q, const double* k, const double* v, int64_t B, int64_t H, int64_t N,
                          int64_t d, double scale) {
  if (!q || !k || !v || B < 1 || H < 1 || N < 1 || d < 1 || !isfinite(scale)) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

/* Forward on fp64 inputs [B,H,N,d] (same definition as oracle_attention_fwd). */
int oracle_attention_fwd_f64(const double* q, const double* k, const double* v, int64_t B, int64_t H, int64_t N,
                             int64_t d, double scale, int causal, double* o_out, double* lse_out) {
  if (check_args_f64(q, k, v, B, H, N, d, scale) || !o_out || !lse_out) return ORACLE_ERR_ARG;
  double* srow = (double*)malloc(sizeof(double) * (size_t)N);
  if (!srow) return ORACLE_ERR_NOMEM;
  for (int64_t bh = 0; bh < B * H; ++bh)
    for (int64_t i = 0; i < N; ++i)
      attention_row(q + (bh * N + i) * d, k + bh * N * d, v + bh * N * d, N, d, scale, causal, i, srow,
                    o_out + (bh * N + i) * d, lse_out + bh * N + i);
  free(srow);
  return ORACLE_OK;
}

/* Backward of one (b,h) slice: q, k, v, dout are N x d; writes dq, dk, dv
 * (N x d) and delta (N). */
/* Row i of the backward: P_i, dP_i, D_i, dS_i and dQ_i (dq_i, d values),
 * with the row statistics m_i, l_i.  p and dp are N-long scratch rows. */
static void bwd_row(const double* q, const double* k, const double* v, const double* dout, int64_t N, int64_t d,
                    double scale, int causal, int64_t i, double* p, double* dp, double* dq_i, double* m_i,
                    double* l_i, double* delta_i) {
  const int64_t nvis = causal ? (i + 1 < N ? i + 1 : N) : N;
  const double* qi = q + i * d;
  const double* doi = dout + i * d;
  double mi = -INFINITY;
  for (int64_t j = 0; j < nvis; ++j) {
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += qi[c] * k[j * d + c];
    p[j] = scale * acc;
    if (p[j] > mi) mi = p[j];
  }
  double li = 0.0;
  for (int64_t j = 0; j < nvis; ++j) { p[j] = exp(p[j] - mi); li += p[j]; }
  for (int64_t j = 0; j < nvis; ++j) p[j] /= li;
  double di = 0.0;
  for (int64_t j = 0; j < nvis; ++j) {
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += doi[c] * v[j * d + c];
    dp[j] = acc;
    di += p[j] * dp[j];
  }
  for (int64_t c = 0; c < d; ++c) dq_i[c] = 0.0;
  for (int64_t j = 0; j < nvis; ++j) {
    const double ds = p[j] * (dp[j] - di);
    for (int64_t c = 0; c < d; ++c) dq_i[c] += scale * ds * k[j * d + c];
  }
  *m_i = mi;
  *l_i = li;
  *delta_i = di;
}

/* Key j of the backward: dK_j and dV_j summed over the rows i that see key j,
 * P_ij and dS_ij rebuilt from the rows' statistics m, l and delta. */
static void bwd_key(const double* q, const double* k, const double* v, const double* dout, int64_t N, int64_t d,
                    double scale, int causal, int64_t j, const double* m, const double* l, const double* delta,
                    double* dk_j, double* dv_j) {
  for (int64_t c = 0; c < d; ++c) { dk_j[c] = 0.0; dv_j[c] = 0.0; }
  for (int64_t i = causal ? j : 0; i < N; ++i) {
    double s = 0.0, dpij = 0.0;
    for (int64_t c = 0; c < d; ++c) {
      s += q[i * d + c] * k[j * d + c];
      dpij += dout[i * d + c] * v[j * d + c];
    }
    const double pij = exp(scale * s - m[i]) / l[i];
    const double ds = pij * (dpij - delta[i]);
    for (int64_t c = 0; c < d; ++c) {
      dv_j[c] += pij * dout[i * d + c];
      dk_j[c] += scale * ds * q[i * d + c];
    }
  }
}

static int attention_bwd_slice(const double* q, const double* k, const double* v, const double* dout, int64_t N,
                               int64_t d, double scale, int causal, double* dq, double* dk, double* dv,
                               double* delta) {
  double* m = (double*)malloc(sizeof(double) * (size_t)N);
  double* l = (double*)malloc(sizeof(double) * (size_t)N);
  if (!m || !l) { free(m); free(l); return ORACLE_ERR_NOMEM; }
  int nomem = 0;
  /* rows: P_i, dP_i, D_i, dS_i, dQ_i */
#pragma omp parallel reduction(| : nomem)
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)N);
    double* dp = (double*)malloc(sizeof(double) * (size_t)N);
    if (!p || !dp) {
      nomem = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t i = 0; i < N; ++i)
        bwd_row(q, k, v, dout, N, d, scale, causal, i, p, dp, dq + i * d, m + i, l + i, delta + i);
    }
    free(p);
    free(dp);
  }
  if (nomem) { free(m); free(l); return ORACLE_ERR_NOMEM; }
  /* keys: dK_j, dV_j over the rows that see key j */
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t j = 0; j < N; ++j) bwd_key(q, k, v, dout, N, d, scale, causal, j, m, l, delta, dk + j * d, dv + j * d);
  free(m);
  free(l);
  return ORACLE_OK;
}

/* Backward on fp64 inputs [B,H,N,d]; outputs dq, dk, dv [B,H,N,d] and
 * delta [B,H,N] (D_i = sum_j P_ij dP_ij). */
int oracle_attention_bwd_f64(const double* q, const double* k, const double* v, const double* dout, int64_t B,
                             int64_t H, int64_t N, int64_t d, double scale, int causal, double* dq, double* dk,
                             double* dv, double* delta, int threads) {
  if (check_args_f64(q, k, v, B, H, N, d, scale) || !dout || !dq || !dk || !dv || !delta) return ORACLE_ERR_ARG;
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
  for (int64_t bh = 0; bh < B * H; ++bh) {
    const int64_t off = bh * N * d;
    int rc = attention_bwd_slice(q + off, k + off, v + off, dout + off, N, d, scale, causal, dq + off, dk + off,
                                 dv + off, delta + bh * N);
    if (rc) return rc;
  }
  return ORACLE_OK;
}

/* Backward on 16-bit inputs (widened exactly first). */
int oracle_attention_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout, int dtype,
                         int64_t B, int64_t H, int64_t N, int64_t d, double scale, int causal, double* dq,
                         double* dk, double* dv, double* delta, int threads) {
  int rc = check_args(q, k, v, dtype, B, H, N, d, scale);
  if (rc) return rc;
  if (!dout) return ORACLE_ERR_ARG;
  const int64_t n = B * H * N * d;
  double* buf = (double*)malloc(sizeof(double) * (size_t)(4 * n));
  if (!buf) return ORACLE_ERR_NOMEM;
  for (int64_t x = 0; x < n; ++x) {
    buf[x] = widen(q[x], dtype);
    buf[n + x] = widen(k[x], dtype);
    buf[2 * n + x] = widen(v[x], dtype);
    buf[3 * n + x] = widen(dout[x], dtype);
  }
  rc = oracle_attention_bwd_f64(buf, buf + n, buf + 2 * n, buf + 3 * n, B, H, N, d, scale, causal, dq, dk, dv,
                                delta, threads);
  free(buf);
  return rc;
}

/* dQ rows and D_i of the backward at sampled (bh, row) pairs, on 16-bit
 * inputs (widened exactly first): the rows pass of the backward above, for
 * the listed rows only.  dq [count, d], delta [count]. */
int oracle_attention_bwd_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                              int dtype, int64_t B, int64_t H, int64_t N, int64_t d, double scale, int causal,
                              const int64_t* bh_idx, const int64_t* row_idx, int64_t count, double* dq,
                              double* delta, int threads) {
  int rc = check_args(q, k, v, dtype, B, H, N, d, scale);
  if (rc) return rc;
  if (!dout || !bh_idx || !row_idx || count < 0 || !dq || !delta) return ORACLE_ERR_ARG;
  for (int64_t s = 0; s < count; ++s)
    if (bh_idx[s] < 0 || bh_idx[s] >= B * H || row_idx[s] < 0 || row_idx[s] >= N) return ORACLE_ERR_ARG;
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
  const int64_t slice = N * d;
  int nomem = 0;
#pragma omp parallel reduction(| : nomem)
  {
    double* buf = (double*)malloc(sizeof(double) * (size_t)(4 * slice + 2 * N));
    if (!buf) {
      nomem = 1;
    } else {
      int64_t have = -1;   /* the (b, h) slice widened in buf */
#pragma omp for schedule(dynamic, 1)
      for (int64_t s = 0; s < count; ++s) {
        const int64_t bh = bh_idx[s];
        if (bh != have) {
          const int64_t off = bh * slice;
          for (int64_t x = 0; x < slice; ++x) {
            buf[x] = widen(q[off + x], dtype);
            buf[slice + x] = widen(k[off + x], dtype);
            buf[2 * slice + x] = widen(v[off + x], dtype);
            buf[3 * slice + x] = widen(dout[off + x], dtype);
          }
          have = bh;
        }
        double m_i, l_i;
        bwd_row(buf, buf + slice, buf + 2 * slice, buf + 3 * slice, N, d, scale, causal, row_idx[s],
                buf + 4 * slice, buf + 4 * slice + N, dq + s * d, &m_i, &l_i, delta + s);
      }
    }
    free(buf);
  }
  return nomem ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* dK and dV rows of the backward at sampled keys of one (b, h) slice bh, on
 * 16-bit inputs: the rows pass for every row that sees one of the keys (with
 * causal masking the rows from the smallest key on), then the keys pass for
 * the listed keys.  dk, dv [count, d]. */
int oracle_attention_bwd_keys(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                              int dtype, int64_t B, int64_t H, int64_t N, int64_t d, double scale, int causal,
                              int64_t bh, const int64_t* key_idx, int64_t count, double* dk, double* dv,
                              int threads) {
  int rc = check_args(q, k, v, dtype, B, H, N, d, scale);
  if (rc) return rc;
  if (!dout || !key_idx || count < 0 || !dk || !dv || bh < 0 || bh >= B * H) return ORACLE_ERR_ARG;
  int64_t first = N;
  for (int64_t s = 0; s < count; ++s) {
    if (key_idx[s] < 0 || key_idx[s] >= N) return ORACLE_ERR_ARG;
    if (key_idx[s] < first) first = key_idx[s];
  }
  const int64_t i0 = causal ? first : 0;   /* rows before i0 see none of the keys */
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
  const int64_t slice = N * d, off = bh * slice;
  double* buf = (double*)malloc(sizeof(double) * (size_t)(4 * slice + 3 * N));
  if (!buf) return ORACLE_ERR_NOMEM;
  double *qd = buf, *kd = buf + slice, *vd = buf + 2 * slice, *dod = buf + 3 * slice;
  double *m = buf + 4 * slice, *l = m + N, *delta = l + N;
  for (int64_t x = 0; x < slice; ++x) {
    qd[x] = widen(q[off + x], dtype);
    kd[x] = widen(k[off + x], dtype);
    vd[x] = widen(v[off + x], dtype);
    dod[x] = widen(dout[off + x], dtype);
  }
  int nomem = 0;
#pragma omp parallel reduction(| : nomem)
  {
    double* scratch = (double*)malloc(sizeof(double) * (size_t)(2 * N + d));
    if (!scratch) {
      nomem = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t i = i0; i < N; ++i)
        bwd_row(qd, kd, vd, dod, N, d, scale, causal, i, scratch, scratch + N, scratch + 2 * N, m + i, l + i,
                delta + i);
    }
    free(scratch);
  }
  if (!nomem) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t s = 0; s < count; ++s)
      bwd_key(qd, kd, vd, dod, N, d, scale, causal, key_idx[s], m, l, delta, dk + s * d, dv + s * d);
  }
  free(buf);
  return nomem ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* ------------------------------------------------------------------ masks and N_q != N_k */

/*
 * Forward with a general mask and separate query / key lengths.  Query i
 * (0 <= i < Nq) and key j (0 <= j < Nk) are aligned at the end of the key
 * sequence (offset off = Nk - Nq, so the last query faces the last key), and
 * key j is visible iff
 *
 *     j < prefix_len                           (keys every query sees), or
 *     j >= i + off - window_left               (when window_left >= 0) and
 *     j <= i + off + window_right              (when window_right >= 0; causal is window_right = 0)
 *
 * -- the additive 0 / -inf mask of the Flash Attention 2 page ("Causal
 * masking", Option A: sliding windows, prefix-LM and the like are a 0/-inf
 * add before softmax).  A row that sees no key has O = 0 and L = -inf.
 */
static int key_visible(int64_t i, int64_t j, int64_t off, int64_t window_left, int64_t window_right,
                       int64_t prefix_len) {
  if (j < prefix_len) return 1;
  if (window_left >= 0 && j < i + off - window_left) return 0;
  if (window_right >= 0 && j > i + off + window_right) return 0;
  return 1;
}

/* One output row by the definition: s_j = scale q.k_j over the visible keys,
 * P = softmax(s), o = sum_j P_j v_j, L = m + ln sum_j exp(s_j - m).  kmat,
 * vmat: [Nk, d] float64; srow: Nk scratch. */
static void masked_row(const double* qrow, const double* kmat, const double* vmat, int64_t i, int64_t Nq, int64_t Nk,
                       int64_t d, double scale, int64_t window_left, int64_t window_right, int64_t prefix_len,
                       double* srow, double* orow, double* lse) {
  const int64_t off = Nk - Nq;
  double m = -INFINITY;
  int64_t seen = 0;
  for (int64_t j = 0; j < Nk; ++j) {
    if (!key_visible(i, j, off, window_left, window_right, prefix_len)) continue;
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += qrow[c] * kmat[j * d + c];
    srow[j] = scale * acc;
    if (srow[j] > m) m = srow[j];
    ++seen;
  }
  for (int64_t c = 0; c < d; ++c) orow[c] = 0.0;
  if (seen == 0) {
    *lse = -INFINITY;
    return;
  }
  double sum = 0.0;
  for (int64_t j = 0; j < Nk; ++j) {
    if (!key_visible(i, j, off, window_left, window_right, prefix_len)) continue;
    srow[j] = exp(srow[j] - m);
    sum += srow[j];
  }
  for (int64_t j = 0; j < Nk; ++j) {
    if (!key_visible(i, j, off, window_left, window_right, prefix_len)) continue;
    const double pj = srow[j] / sum;
    for (int64_t c = 0; c < d; ++c) orow[c] += pj * vmat[j * d + c];
  }
  *lse = m + log(sum);
}

static int masked_args_ok(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype, int64_t B, int64_t H,
                          int64_t Nq, int64_t Nk, int64_t d, double scale, int64_t prefix_len) {
  if (!q || !k || !v || (dtype != ORACLE_FP16 && dtype != ORACLE_BF16)) return 0;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1 || !isfinite(scale) || prefix_len < 0) return 0;
  return 1;
}

/* q: [B,H,Nq,d], k, v: [B,H,Nk,d] (16-bit bit patterns); o: [B,H,Nq,d], lse: [B,H,Nq]. */
int oracle_attention_fwd_masked(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype, int64_t B,
                                int64_t H, int64_t Nq, int64_t Nk, int64_t d, double scale, int64_t window_left,
                                int64_t window_right, int64_t prefix_len, double* o_out, double* lse_out,
                                int threads) {
  if (!masked_args_ok(q, k, v, dtype, B, H, Nq, Nk, d, scale, prefix_len) || !o_out || !lse_out)
    return ORACLE_ERR_ARG;
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
  double* kmat = (double*)malloc(sizeof(double) * (size_t)(Nk * d));
  double* vmat = (double*)malloc(sizeof(double) * (size_t)(Nk * d));
  if (!kmat || !vmat) { free(kmat); free(vmat); return ORACLE_ERR_NOMEM; }
  int status = ORACLE_OK;
  for (int64_t bh = 0; bh < B * H && status == ORACLE_OK; ++bh) {
    for (int64_t x = 0; x < Nk * d; ++x) {
      kmat[x] = widen(k[bh * Nk * d + x], dtype);
      vmat[x] = widen(v[bh * Nk * d + x], dtype);
    }
    int nomem = 0;
#pragma omp parallel reduction(| : nomem)
    {
      double* srow = (double*)malloc(sizeof(double) * (size_t)Nk);
      double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
      if (!srow || !qrow) {
        nomem = 1;
      } else {
#pragma omp for schedule(dynamic, 4)
        for (int64_t i = 0; i < Nq; ++i) {
          for (int64_t c = 0; c < d; ++c) qrow[c] = widen(q[(bh * Nq + i) * d + c], dtype);
          masked_row(qrow, kmat, vmat, i, Nq, Nk, d, scale, window_left, window_right, prefix_len, srow,
                     o_out + (bh * Nq + i) * d, lse_out + bh * Nq + i);
        }
      }
      free(srow);
      free(qrow);
    }
    if (nomem) status = ORACLE_ERR_NOMEM;
  }
  free(kmat);
  free(vmat);
  return status;
}

/* The same definition at sampled (bh, row) pairs only: o: [count, d],
 * lse: [count].  For problems too large to evaluate whole. */
int oracle_attention_rows_masked(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype, int64_t B,
                                 int64_t H, int64_t Nq, int64_t Nk, int64_t d, double scale, int64_t window_left,
                                 int64_t window_right, int64_t prefix_len, const int64_t* bh_idx,
                                 const int64_t* row_idx, int64_t count, double* o_out, double* lse_out,
                                 int threads) {
  if (!masked_args_ok(q, k, v, dtype, B, H, Nq, Nk, d, scale, prefix_len) || !o_out || !lse_out || count < 0 ||
      (count > 0 && (!bh_idx || !row_idx)))
    return ORACLE_ERR_ARG;
  for (int64_t s = 0; s < count; ++s)
    if (bh_idx[s] < 0 || bh_idx[s] >= B * H || row_idx[s] < 0 || row_idx[s] >= Nq) return ORACLE_ERR_ARG;
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
  int nomem = 0;
#pragma omp parallel reduction(| : nomem)
  {
    double* kmat = (double*)malloc(sizeof(double) * (size_t)(Nk * d));
    double* vmat = (double*)malloc(sizeof(double) * (size_t)(Nk * d));
    double* srow = (double*)malloc(sizeof(double) * (size_t)Nk);
    double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
    int64_t have = -1;  /* the (b,h) whose K and V are widened in kmat / vmat */
    if (!kmat || !vmat || !srow || !qrow) {
      nomem = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t s = 0; s < count; ++s) {
        const int64_t bh = bh_idx[s], i = row_idx[s];
        if (bh != have) {
          for (int64_t x = 0; x < Nk * d; ++x) {
            kmat[x] = widen(k[bh * Nk * d + x], dtype);
            vmat[x] = widen(v[bh * Nk * d + x], dtype);
          }
          have = bh;
        }
        for (int64_t c = 0; c < d; ++c) qrow[c] = widen(q[(bh * Nq + i) * d + c], dtype);
        masked_row(qrow, kmat, vmat, i, Nq, Nk, d, scale, window_left, window_right, prefix_len, srow,
                   o_out + s * d, lse_out + s);
      }
    }
    free(kmat);
    free(vmat);
    free(srow);
    free(qrow);
  }
  return nomem ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* ------------------------------------------------------------------ masked backward */

/*
 * Gradients of the masked forward above (FlashAttention V2 in depth,
 * section 7: P = softmax over the visible keys, dV = P^T dO, dP = dO V^T,
 * D_i = rowsum(dO_i o O_i) = sum_j P_ij dP_ij, dS = P o (dP - D),
 * dQ = scale dS K, dK = scale dS^T Q), for one (b,h) slice of float64 data:
 * q, dout [Nq,d], k, v [Nk,d].  Hidden pairs contribute nothing; a row that
 * sees no key has dQ = 0 and D = 0; a key no row sees has dK = dV = 0.
 */
static int masked_bwd_slice(const double* q, const double* k, const double* v, const double* dout, int64_t Nq,
                            int64_t Nk, int64_t d, double scale, int64_t wl, int64_t wr, int64_t prefix,
                            double* dq, double* dk, double* dv, double* delta) {
  const int64_t off = Nk - Nq;
  double* m = (double*)malloc(sizeof(double) * (size_t)Nq);
  double* l = (double*)malloc(sizeof(double) * (size_t)Nq);
  if (!m || !l) { free(m); free(l); return ORACLE_ERR_NOMEM; }
  int nomem = 0;
  /* rows: m_i, l_i, D_i, dQ_i */
#pragma omp parallel reduction(| : nomem)
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)Nk);
    if (!s) {
      nomem = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t i = 0; i < Nq; ++i) {
        const double* qi = q + i * d;
        const double* doi = dout + i * d;
        double mi = -INFINITY;
        for (int64_t j = 0; j < Nk; ++j) {
          if (!key_visible(i, j, off, wl, wr, prefix)) continue;
          double acc = 0.0;
          for (int64_t c = 0; c < d; ++c) acc += qi[c] * k[j * d + c];
          s[j] = scale * acc;
          if (s[j] > mi) mi = s[j];
        }
        for (int64_t c = 0; c < d; ++c) dq[i * d + c] = 0.0;
        m[i] = mi;
        l[i] = 0.0;
        delta[i] = 0.0;
        if (mi == -INFINITY) continue;
        double li = 0.0;
        for (int64_t j = 0; j < Nk; ++j)
          if (key_visible(i, j, off, wl, wr, prefix)) li += exp(s[j] - mi);
        double di = 0.0;
        for (int64_t j = 0; j < Nk; ++j) {
          if (!key_visible(i, j, off, wl, wr, prefix)) continue;
          double dp = 0.0;
          for (int64_t c = 0; c < d; ++c) dp += doi[c] * v[j * d + c];
          di += exp(s[j] - mi) / li * dp;
        }
        for (int64_t j = 0; j < Nk; ++j) {
          if (!key_visible(i, j, off, wl, wr, prefix)) continue;
          double dp = 0.0;
          for (int64_t c = 0; c < d; ++c) dp += doi[c] * v[j * d + c];
          const double ds = exp(s[j] - mi) / li * (dp - di);
          for (int64_t c = 0; c < d; ++c) dq[i * d + c] += scale * ds * k[j * d + c];
        }
        l[i] = li;
        delta[i] = di;
      }
    }
    free(s);
  }
  if (nomem) { free(m); free(l); return ORACLE_ERR_NOMEM; }
  /* keys: dK_j, dV_j over the rows that see key j */
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t j = 0; j < Nk; ++j) {
    for (int64_t c = 0; c < d; ++c) { dk[j * d + c] = 0.0; dv[j * d + c] = 0.0; }
    for (int64_t i = 0; i < Nq; ++i) {
      if (!key_visible(i, j, off, wl, wr, prefix) || m[i] == -INFINITY) continue;
      double sij = 0.0, dpij = 0.0;
      for (int64_t c = 0; c < d; ++c) {
        sij += q[i * d + c] * k[j * d + c];
        dpij += dout[i * d + c] * v[j * d + c];
      }
      const double pij = exp(scale * sij - m[i]) / l[i];
      const double ds = pij * (dpij - delta[i]);
      for (int64_t c = 0; c < d; ++c) {
        dv[j * d + c] += pij * dout[i * d + c];
        dk[j * d + c] += scale * ds * q[i * d + c];
      }
    }
  }
  free(m);
  free(l);
  return ORACLE_OK;
}

static int masked_f64_args_ok(const double* q, const double* k, const double* v, int64_t B, int64_t H, int64_t Nq,
                              int64_t Nk, int64_t d, double scale, int64_t prefix_len) {
  if (!q || !k || !v) return 0;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1 || !isfinite(scale) || prefix_len < 0) return 0;
  return 1;
}

/* The masked forward on float64 inputs q [B,H,Nq,d], k, v [B,H,Nk,d]. */
int oracle_attention_fwd_masked_f64(const double* q, const double* k, const double* v, int64_t B, int64_t H,
                                    int64_t Nq, int64_t Nk, int64_t d, double scale, int64_t window_left,
                                    int64_t window_right, int64_t prefix_len, double* o_out, double* lse_out) {
  if (!masked_f64_args_ok(q, k, v, B, H, Nq, Nk, d, scale, prefix_len) || !o_out || !lse_out) return ORACLE_ERR_ARG;
  double* srow = (double*)malloc(sizeof(double) * (size_t)Nk);
  if (!srow) return ORACLE_ERR_NOMEM;
  for (int64_t bh = 0; bh < B * H; ++bh)
    for (int64_t i = 0; i < Nq; ++i)
      masked_row(q + (bh * Nq + i) * d, k + bh * Nk * d, v + bh * Nk * d, i, Nq, Nk, d, scale, window_left,
                 window_right, prefix_len, srow, o_out + (bh * Nq + i) * d, lse_out + bh * Nq + i);
  free(srow);
  return ORACLE_OK;
}

/* Masked backward on float64 inputs: dq, dout [B,H,Nq,d]; dk, dv [B,H,Nk,d]; delta [B,H,Nq]. */
int oracle_attention_bwd_masked_f64(const double* q, const double* k, const double* v, const double* dout, int64_t B,
                                    int64_t H, int64_t Nq, int64_t Nk, int64_t d, double scale, int64_t window_left,
                                    int64_t window_right, int64_t prefix_len, double* dq, double* dk, double* dv,
                                    double* delta, int threads) {
  if (!masked_f64_args_ok(q, k, v, B, H, Nq, Nk, d, scale, prefix_len) || !dout || !dq || !dk || !dv || !delta)
    return ORACLE_ERR_ARG;
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
  for (int64_t bh = 0; bh < B * H; ++bh) {
    const int64_t oq = bh * Nq * d, ok = bh * Nk * d;
    int rc = masked_bwd_slice(q + oq, k + ok, v + ok, dout + oq, Nq, Nk, d, scale, window_left, window_right,
                              prefix_len, dq + oq, dk + ok, dv + ok, delta + bh * Nq);
    if (rc) return rc;
  }
  return ORACLE_OK;
}

/* Masked backward on 16-bit inputs (widened exactly first). */
int oracle_attention_bwd_masked(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                                int dtype, int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, double scale,
                                int64_t window_left, int64_t window_right, int64_t prefix_len, double* dq,
                                double* dk, double* dv, double* delta, int threads) {
  if (!masked_args_ok(q, k, v, dtype, B, H, Nq, Nk, d, scale, prefix_len) || !dout) return ORACLE_ERR_ARG;
  const int64_t nq = B * H * Nq * d, nk = B * H * Nk * d;
  double* buf = (double*)malloc(sizeof(double) * (size_t)(2 * nq + 2 * nk));
  if (!buf) return ORACLE_ERR_NOMEM;
  double *bq = buf, *bdo = buf + nq, *bk = buf + 2 * nq, *bv = buf + 2 * nq + nk;
  for (int64_t x = 0; x < nq; ++x) {
    bq[x] = widen(q[x], dtype);
    bdo[x] = widen(dout[x], dtype);
  }
  for (int64_t x = 0; x < nk; ++x) {
    bk[x] = widen(k[x], dtype);
    bv[x] = widen(v[x], dtype);
  }
  int rc = oracle_attention_bwd_masked_f64(bq, bk, bv, bdo, B, H, Nq, Nk, d, scale, window_left, window_right,
                                           prefix_len, dq, dk, dv, delta, threads);
  free(buf);
  return rc;
}

/* Threads OpenMP will use (1 without OpenMP); reported by the CPU baseline. */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
