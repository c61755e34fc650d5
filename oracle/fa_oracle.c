/*
 * fa_oracle.c -- float64 CPU oracle for the FlashAttention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check of the package entry
 * point and the benchmark's CPU-baseline leg use it.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it computes (the plain definition, no tiling, no online rescaling):
 * the reference scaled dot-product attention that the Ascend FlashAttention
 * page verifies its kernel against ("ops-transformer FlashAttention build
 * and tuning", section 4.3, compute_reference_attention): scores are the
 * scaled product Q K^T, the causal variant fills the strict upper triangle
 * (triu with diagonal=1, i.e. column j > row i) with -inf, a row-wise
 * softmax follows, and the result is P V.  The same page (preface) states
 * that FlashAttention is numerically equivalent to this standard attention,
 * so the tiled method reaches exactly this result up to rounding order.
 * Section 6.2 of that page adds the max-subtraction ("safe softmax") step
 * used below so that exp() never overflows; it does not change the value.
 *
 * For each selected query row i of head (b, h):
 *   1. S[j]   = scale * sum_d q[i,d] * k[j,d]            for allowed j
 *   2. allowed set: every j < S_kv; with causal, only j <= i (top-left
 *      alignment, the verifier's triu(diagonal=1) mask)
 *   3. m      = max_{allowed j} S[j]
 *      P[j]   = exp(S[j] - m) / sum_{allowed} exp(S[j'] - m); P[j] = 0 if masked
 *   4. O[i,:] = sum_j P[j] * v[j,:]
 *   5. lse_i  = m + log(sum_{allowed} exp(S[j] - m))      (natural log)
 * S and P are materialised for the whole row (length S_kv) in float64.
 *
 * Inputs are the raw element buffers the GPU consumes: IEEE binary16,
 * bfloat16 or OCP FP8 E4M3 (the "fn" variant: no infinities, one NaN
 * mantissa pattern, max finite 448), decoded here from the format
 * definitions into float64.  For E4M3 the decoded value is multiplied by the
 * per-tensor descale (dq, dk, dv), which is how the Hygon retrospective
 * (defect 17) describes FP8 attention scales: one scalar per tensor.
 *
 * Layouts: BNSD = [B, H, S, D] and BSND = [B, S, H, D], both contiguous;
 * element offsets are 64-bit throughout.
 *
 * Grouped-query attention (the Hygon retrospective, defect 12): Q has H heads,
 * K and V have H_kv heads with H a multiple of H_kv, ngroups = H / H_kv, and
 * query head h reads key/value head h / ngroups (Q viewed as
 * [.., H_kv, ngroups, D] in its own flat head order).  H_kv = H is plain
 * multi-head attention.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };
enum { ORC_BNSD = 0, ORC_BSND = 1 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t x) {
  int sign = (x >> 15) & 1;
  int e = (x >> 10) & 0x1f;
  int f = x & 0x3ff;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -24);             /* subnormal: f * 2^-14 * 2^-10 */
  } else if (e == 31) {
    mag = f ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static double decode_bf16(uint16_t x) {
  int sign = (x >> 15) & 1;
  int e = (x >> 7) & 0xff;
  int f = x & 0x7f;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -133);            /* f * 2^-126 * 2^-7 */
  } else if (e == 255) {
    mag = f ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(128 + f), e - 134); /* (1 + f/128) * 2^(e-127) */
  }
  return sign ? -mag : mag;
}

/* OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent bits (bias 7), 3 fraction bits;
 * exponent 15 with fraction 7 is NaN, there is no infinity. */
static double decode_e4m3(uint8_t x) {
  int sign = (x >> 7) & 1;
  int e = (x >> 3) & 0xf;
  int f = x & 0x7;
  double mag;
  if (e == 15 && f == 7) {
    mag = NAN;
  } else if (e == 0) {
    mag = ldexp((double)f, -9);              /* f * 2^-6 * 2^-3 */
  } else {
    mag = ldexp((double)(8 + f), e - 10);    /* (1 + f/8) * 2^(e-7) */
  }
  return sign ? -mag : mag;
}

static double decode_one(const void* base, int dtype, int64_t idx) {
  switch (dtype) {
    case ORC_F16: return decode_f16(((const uint16_t*)base)[idx]);
    case ORC_BF16: return decode_bf16(((const uint16_t*)base)[idx]);
    default: return decode_e4m3(((const uint8_t*)base)[idx]);
  }
}

/* Offset of element (b, h, s, d) of a [B,H,S,D] or [B,S,H,D] tensor. */
static int64_t elem_offset(int layout, int64_t H, int64_t S, int64_t D,
                           int64_t b, int64_t h, int64_t s, int64_t d) {
  if (layout == ORC_BNSD) return ((b * H + h) * S + s) * D + d;
  return ((b * S + s) * H + h) * D + d;
}

typedef struct {
  const void *q, *k, *v;
  int dtype, layout;
  int64_t B, H, S_q, S_kv, D;
  double scale, dq, dk, dv;
  int causal;
  int64_t H_kv;
} problem_t;

/* Decode row s of head (b, h) of one tensor with `heads` heads into out[0..D). */
static void load_row(const problem_t* p, const void* t, int64_t heads, int64_t S, double ds,
                     int64_t b, int64_t h, int64_t s, double* out) {
  for (int64_t d = 0; d < p->D; ++d) {
    double x = decode_one(t, p->dtype, elem_offset(p->layout, heads, S, p->D, b, h, s, d));
    out[d] = (p->dtype == ORC_E4M3) ? x * ds : x;
  }
}

/* Steps 1-5 above for one query row.  kd, vd hold the decoded K and V of the
 * head, [S_kv, D] row-major; Srow and Prow are S_kv scratch rows. */
static void attend_row(const problem_t* p, const double* qrow, const double* kd,
                       const double* vd, int64_t i, double* Srow, double* Prow,
                       double* o, double* lse) {
  const int64_t S_kv = p->S_kv, D = p->D;
  double m = -INFINITY;
  for (int64_t j = 0; j < S_kv; ++j) {
    int allowed = !p->causal || j <= i;
    if (!allowed) { Srow[j] = -INFINITY; continue; }
    double acc = 0.0;
    for (int64_t d = 0; d < D; ++d) acc += qrow[d] * kd[j * D + d];
    Srow[j] = p->scale * acc;
    if (Srow[j] > m) m = Srow[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < S_kv; ++j) {
    int allowed = !p->causal || j <= i;
    Prow[j] = allowed ? exp(Srow[j] - m) : 0.0;
    l += Prow[j];
  }
  for (int64_t j = 0; j < S_kv; ++j) Prow[j] /= l;
  for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
  for (int64_t j = 0; j < S_kv; ++j) {
    if (Prow[j] == 0.0) continue;  /* masked (or underflowed) weights add nothing */
    for (int64_t d = 0; d < D; ++d) o[d] += Prow[j] * vd[j * D + d];
  }
  *lse = m + log(l);
}

static int check_problem(const problem_t* p) {
  if (!p->q || !p->k || !p->v) return 1;
  if (p->B < 1 || p->H < 1 || p->S_q < 1 || p->S_kv < 1 || p->D < 1) return 2;
  if (p->dtype < ORC_F16 || p->dtype > ORC_E4M3) return 3;
  if (p->layout != ORC_BNSD && p->layout != ORC_BSND) return 4;
  if (p->H_kv < 1 || p->H % p->H_kv != 0) return 8;
  return 0;
}

/* Decode n raw elements of the given type into float64 (no descale). */
int fa_oracle_decode(const void* x, int dtype, int64_t n, double* out) {
  if (!x || !out || n < 0 || dtype < ORC_F16 || dtype > ORC_E4M3) return 1;
  for (int64_t i = 0; i < n; ++i) out[i] = decode_one(x, dtype, i);
  return 0;
}

/* Selected rows: rows holds n_rows triples (b, h, i).  O is [n_rows, D],
 * lse is [n_rows], P (optional, may be NULL) is [n_rows, S_kv].  Each row
 * decodes its own head's K and V, so this suits sparse samples. */
int fa_oracle_rows_gqa(const void* q, const void* k, const void* v, int dtype, int layout,
                       int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv,
                       int64_t D, double scale, int causal, double dq, double dk, double dv,
                       int64_t n_rows, const int64_t* rows, double* O, double* lse,
                       double* P, int n_threads) {
  problem_t p = {q, k, v, dtype, layout, B, H, S_q, S_kv, D, scale, dq, dk, dv, causal, H_kv};
  int rc = check_problem(&p);
  if (rc) return rc;
  if (!rows || !O || !lse || n_rows < 0) return 5;
  for (int64_t r = 0; r < n_rows; ++r) {
    if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 || rows[3 * r + 1] >= H ||
        rows[3 * r + 2] < 0 || rows[3 * r + 2] >= S_q)
      return 6;
  }
  int bad = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
  {
    double* kd = (double*)malloc(sizeof(double) * (size_t)(S_kv * D));
    double* vd = (double*)malloc(sizeof(double) * (size_t)(S_kv * D));
    double* qrow = (double*)malloc(sizeof(double) * (size_t)D);
    double* Srow = (double*)malloc(sizeof(double) * (size_t)S_kv);
    double* Prow = (double*)malloc(sizeof(double) * (size_t)S_kv);
    if (!kd || !vd || !qrow || !Srow || !Prow) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      bad = 1;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int64_t r = 0; r < n_rows; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        int64_t hk = h / (H / H_kv);
        for (int64_t j = 0; j < S_kv; ++j) {
          load_row(&p, k, H_kv, S_kv, dk, b, hk, j, kd + j * D);
          load_row(&p, v, H_kv, S_kv, dv, b, hk, j, vd + j * D);
        }
        load_row(&p, q, H, S_q, dq, b, h, i, qrow);
        attend_row(&p, qrow, kd, vd, i, Srow, Prow, O + r * D, lse + r);
        if (P) memcpy(P + r * S_kv, Prow, sizeof(double) * (size_t)S_kv);
      }
    }
    free(kd); free(vd); free(qrow); free(Srow); free(Prow);
  }
  return bad ? 7 : 0;
}

/* Every row of every head.  O is [B, H, S_q, D] (BNSD, whatever the input
 * layout), lse is [B, H, S_q].  Heads are taken one after another; inside a
 * head the K/V decode and then the query rows run in parallel. */
int fa_oracle_full_gqa(const void* q, const void* k, const void* v, int dtype, int layout,
                       int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv,
                       int64_t D, double scale, int causal, double dq, double dk, double dv,
                       double* O, double* lse, int n_threads) {
  problem_t p = {q, k, v, dtype, layout, B, H, S_q, S_kv, D, scale, dq, dk, dv, causal, H_kv};
  int rc = check_problem(&p);
  if (rc) return rc;
  if (!O || !lse) return 5;
  double* kd = (double*)malloc(sizeof(double) * (size_t)(S_kv * D));
  double* vd = (double*)malloc(sizeof(double) * (size_t)(S_kv * D));
  if (!kd || !vd) { free(kd); free(vd); return 7; }
  int bad = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#endif
  for (int64_t bh = 0; bh < B * H && !bad; ++bh) {
    const int64_t b = bh / H, h = bh % H, hk = h / (H / H_kv);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t j = 0; j < S_kv; ++j) {
      load_row(&p, k, H_kv, S_kv, dk, b, hk, j, kd + j * D);
      load_row(&p, v, H_kv, S_kv, dv, b, hk, j, vd + j * D);
    }
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
      double* qrow = (double*)malloc(sizeof(double) * (size_t)D);
      double* Srow = (double*)malloc(sizeof(double) * (size_t)S_kv);
      double* Prow = (double*)malloc(sizeof(double) * (size_t)S_kv);
      if (!qrow || !Srow || !Prow) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
        bad = 1;
      } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (int64_t i = 0; i < S_q; ++i) {
          load_row(&p, q, H, S_q, dq, b, h, i, qrow);
          attend_row(&p, qrow, kd, vd, i, Srow, Prow, O + (bh * S_q + i) * D, lse + bh * S_q + i);
        }
      }
      free(qrow); free(Srow); free(Prow);
    }
  }
  free(kd); free(vd);
  return bad ? 7 : 0;
}

/* Multi-head attention: the grouped entry points with H_kv = H. */
int fa_oracle_rows(const void* q, const void* k, const void* v, int dtype, int layout,
                   int64_t B, int64_t H, int64_t S_q, int64_t S_kv, int64_t D,
                   double scale, int causal, double dq, double dk, double dv,
                   int64_t n_rows, const int64_t* rows, double* O, double* lse,
                   double* P, int n_threads) {
  return fa_oracle_rows_gqa(q, k, v, dtype, layout, B, H, H, S_q, S_kv, D, scale, causal, dq, dk,
                            dv, n_rows, rows, O, lse, P, n_threads);
}

int fa_oracle_full(const void* q, const void* k, const void* v, int dtype, int layout,
                   int64_t B, int64_t H, int64_t S_q, int64_t S_kv, int64_t D,
                   double scale, int causal, double dq, double dk, double dv,
                   double* O, double* lse, int n_threads) {
  return fa_oracle_full_gqa(q, k, v, dtype, layout, B, H, H, S_q, S_kv, D, scale, causal, dq, dk,
                            dv, O, lse, n_threads);
}

/* Threads an OpenMP region would use (1 without OpenMP). */
int fa_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
