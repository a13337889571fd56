/*
 * dsa_oracle.c -- plain, slow, obviously-correct CPU oracle of the DSA hot path
 * (Lightning Indexer scoring + top-K selection, then Sparse Flash Attention over the
 * selected positions), in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this file:
 * only the tests, the package smoke check and the benchmark's CPU-baseline leg do.  It shares
 * no code, header, table or constant generator with the CUDA library; both sides read the same
 * input bytes and nothing else.
 *
 * What it follows (the public pages on Kimi K3.1 Pro inference, DSA path):
 *   - "Inference Optimization for Kimi K3.1 Pro: Decoding Architecture Evolution and Systems
 *     Engineering Practices", section 1 (Algorithmic Architecture Analysis), the three DSA steps:
 *     the indexer scores each historical key against the current query with head weights, the
 *     top K positions are kept, and sparse attention reads only those positions.
 *   - same page, section 2 (Operator-Level Deep Fusion): the score / head-weight / top-K fusion
 *     changes where intermediates live, not the result -- so the oracle computes the plain,
 *     unfused definition.
 *   - "Optimizing Kimi K3.1 Pro Sparse Attention Inference: Day0 Adaptation and Performance
 *     Tuning on Ascend", section "Inheritance and Extension of Core Operators": SFA is exact
 *     attention over the gathered rows, computed blockwise on the device; the oracle computes the
 *     same softmax directly (not blockwise).
 *   - "Day0 Inference Adaptation for Next-Gen LLMs ... CANN", section 3.1: the indexer reads a
 *     paged key cache, SFA reads the main attention (latent) cache at the selected indices.
 *
 * Readings where the pages are silent (stated here and listed in the design notes):
 *   score      s(t,j) = sum_h w[t,h] * max(0, q[t,h,:] . k[j,:]); one key row per position,
 *              shared by all index heads; for e4m3 inputs q and k are the dequantised values
 *              q8 * q_scale[t,h] and k8 * k_scale[row]; for MXFP8 inputs ("Inference
 *              Optimization for Kimi K3.1 Pro", section 4, fully quantised indexer path; "Day0
 *              Inference Adaptation ... CANN", section 3.3: group size 32) every run of 32
 *              consecutive elements of a q head or a key row shares one power-of-two scale, so
 *              the dequantised value of element d is e4m3(q8[d]) * 2^(sf[d / 32] - 127).
 *   visibility a query token at absolute position p sees positions 0..p (itself included);
 *              the n new tokens of a sequence of length L sit at L-n .. L-1.
 *   selection  the first min(K, p+1) positions in the order (score descending, position
 *              ascending); emitted in ascending position order, then -1 padding.
 *   attention  z_j = scale * q[t,h,0:576] . kv[j,0:576];  o = sum_j softmax(z)_j kv[j,0:512];
 *              lse = max z + log(sum exp(z - max z)) (natural log).  An empty index set gives
 *              o = 0 and lse = -inf.
 *
 * Parity pins (tests/test_oracle.py) tie each function to something other than itself: a
 * hand-worked example, closed forms, library routines (torch's fp8/bf16 decoders and dense
 * attention), brute-force validity of the selection, and page-table permutation invariance.
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -fPIC -shared (see oracle/build.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EARG (-1)
#define ORC_EINDEX (-2)
#define ORC_ENOMEM (-3)

typedef struct {
  int B, n_q, H_I, d_I, K, page_size, max_pages, num_pages;
  int fp8;                    /* 0: bf16 q/k; 1: e4m3 q/k with fp32 scales;
                                 2: MXFP8 (e4m3 q/k with E8M0 scales per 32 elements)    */
  const void* q;              /* [n_q][H_I][d_I]                                        */
  const float* q_scale;       /* [n_q][H_I]          (fp8 only)                         */
  const float* w;             /* [n_q][H_I]                                             */
  const void* k_pool;         /* [num_pages][page_size][d_I]                            */
  const float* k_scale;       /* [num_pages][page_size] (fp8 only)                      */
  const int* page_table;      /* [B][max_pages]                                         */
  const int* seq_lens;        /* [B]                                                    */
  const int* q_start;         /* [B+1]                                                  */
  const uint8_t* q_sf;        /* [n_q][H_I][d_I/32] E8M0   (MXFP8 only)                 */
  const uint8_t* k_sf;        /* [num_pages][page_size][d_I/32] E8M0 (MXFP8 only)       */
} orc_li;

typedef struct {
  int B, n_q, H, d_qk, d_v, K, page_size, max_pages, num_pages;
  double scale;
  const uint16_t* q;          /* [n_q][H][d_qk] bf16 bits                               */
  const uint16_t* kv_pool;    /* [num_pages][page_size][d_qk] bf16 bits                 */
  const int* page_table;      /* [B][max_pages]                                         */
  const int* seq_lens;        /* [B]                                                    */
  const int* q_start;         /* [B+1]                                                  */
} orc_sfa;

/* ---- number formats, from their definitions ------------------------------------------ */

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
double orc_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
 * subnormals when the exponent field is 0, no infinities, NaN = S.1111.111. */
double orc_e4m3(uint8_t bits) {
  int s = (bits >> 7) & 1, e = (bits >> 3) & 15, m = bits & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* OCP Microscaling E8M0 scale: an unsigned 8-bit exponent with bias 127, value 2^(e - 127);
 * 0xFF is NaN. */
double orc_e8m0(uint8_t bits) {
  if (bits == 0xFF) return NAN;
  return ldexp(1.0, (int)bits - 127);
}

/* ---- token -> (sequence, position) and position -> physical row ---------------------- */

static int locate(const int* q_start, const int* seq_lens, int B, int t, int* b_out, int* p_out) {
  for (int b = 0; b < B; ++b) {
    if (t >= q_start[b] && t < q_start[b + 1]) {
      int n_new = q_start[b + 1] - q_start[b];
      int p = seq_lens[b] - n_new + (t - q_start[b]);
      if (p < 0) return ORC_EARG;
      *b_out = b;
      *p_out = p;
      return ORC_OK;
    }
  }
  return ORC_EARG;
}

static long long phys_row(const int* pt, int max_pages, int page_size, int b, int j) {
  return (long long)pt[(long long)b * max_pages + j / page_size] * page_size + j % page_size;
}

/* ---- Lightning Indexer scores -------------------------------------------------------- */

static double li_q(const orc_li* P, int t, int h, int d) {
  long long i = ((long long)t * P->H_I + h) * P->d_I + d;
  if (P->fp8 == 2)
    return orc_e4m3(((const uint8_t*)P->q)[i]) *
           orc_e8m0(P->q_sf[((long long)t * P->H_I + h) * (P->d_I / 32) + d / 32]);
  if (P->fp8) return orc_e4m3(((const uint8_t*)P->q)[i]) * (double)P->q_scale[(long long)t * P->H_I + h];
  return orc_bf16(((const uint16_t*)P->q)[i]);
}

static double li_k(const orc_li* P, long long row, int d) {
  long long i = row * P->d_I + d;
  if (P->fp8 == 2) return orc_e4m3(((const uint8_t*)P->k_pool)[i]) * orc_e8m0(P->k_sf[row * (P->d_I / 32) + d / 32]);
  if (P->fp8) return orc_e4m3(((const uint8_t*)P->k_pool)[i]) * (double)P->k_scale[row];
  return orc_bf16(((const uint16_t*)P->k_pool)[i]);
}

/* s(t, j) and a bound on sum_h |w_h| sum_d |q_hd k_jd| (the magnitude any fp32 evaluation's
 * rounding error is proportional to). */
static double li_score(const orc_li* P, int t, int b, int j, double* mag) {
  long long row = phys_row(P->page_table, P->max_pages, P->page_size, b, j);
  double s = 0.0, m = 0.0;
  for (int h = 0; h < P->H_I; ++h) {
    double dot = 0.0, adot = 0.0;
    for (int d = 0; d < P->d_I; ++d) {
      double prod = li_q(P, t, h, d) * li_k(P, row, d);
      dot += prod;
      adot += fabs(prod);
    }
    double wh = (double)P->w[(long long)t * P->H_I + h];
    s += wh * (dot > 0.0 ? dot : 0.0);
    m += fabs(wh) * adot;
  }
  if (mag) *mag = m;
  return s;
}

static int li_check(const orc_li* P) {
  if (!P || P->B <= 0 || P->n_q < 0 || P->H_I <= 0 || P->d_I <= 0 || P->K <= 0 ||
      P->page_size <= 0 || P->max_pages <= 0 || !P->q || !P->w || !P->k_pool ||
      !P->page_table || !P->seq_lens || !P->q_start)
    return ORC_EARG;
  if (P->fp8 == 1 && (!P->q_scale || !P->k_scale)) return ORC_EARG;
  if (P->fp8 == 2 && (!P->q_sf || !P->k_sf || P->d_I % 32 != 0)) return ORC_EARG;
  if (P->fp8 < 0 || P->fp8 > 2) return ORC_EARG;
  for (int b = 0; b < P->B; ++b) {
    int L = P->seq_lens[b];
    if (L < 0 || (L + P->page_size - 1) / P->page_size > P->max_pages) return ORC_EARG;
    for (int p = 0; p < (L + P->page_size - 1) / P->page_size; ++p) {
      int pg = P->page_table[(long long)b * P->max_pages + p];
      if (pg < 0 || pg >= P->num_pages) return ORC_EARG;
    }
  }
  return ORC_OK;
}

/* Scores of token t for all visible positions 0..p; returns p+1 (or a negative error). */
int oracle_li_scores(const orc_li* P, int t, double* s_out, double* mag_out) {
  int rc = li_check(P), b, p;
  if (rc) return rc;
  if ((rc = locate(P->q_start, P->seq_lens, P->B, t, &b, &p))) return rc;
  for (int j = 0; j <= p; ++j) s_out[j] = li_score(P, t, b, j, mag_out ? &mag_out[j] : NULL);
  return p + 1;
}

typedef struct { double s; int j; } cand;

/* Selection order: larger score first; equal scores -> lower position first.  Real-valued
 * comparison, so -0.0 and +0.0 are equal. */
static int by_score_then_pos(const void* a, const void* b) {
  const cand* x = (const cand*)a;
  const cand* y = (const cand*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->j > y->j) - (x->j < y->j);
}

static int by_int(const void* a, const void* b) {
  int x = *(const int*)a, y = *(const int*)b;
  return (x > y) - (x < y);
}

/* Top-K of each listed token by a full sort: out_idx[i][0..K) ascending positions, -1 padded;
 * out_cnt[i] = min(K, p+1); out_kth[i] (optional) = score of the last selected position in
 * selection order (the K-th largest). */
int oracle_li_topk(const orc_li* P, int n_tok, const int* toks, int* out_idx, int* out_cnt,
                   double* out_kth) {
  int rc = li_check(P);
  if (rc) return rc;
  if (n_tok < 0 || (n_tok > 0 && (!toks || !out_idx))) return ORC_EARG;
  for (int i = 0; i < n_tok; ++i) {
    int b, p;
    if (toks[i] < 0 || toks[i] >= P->n_q) return ORC_EARG;
    if (locate(P->q_start, P->seq_lens, P->B, toks[i], &b, &p)) return ORC_EARG;
  }
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n_tok; ++i) {
    int t = toks[i], b, p;
    locate(P->q_start, P->seq_lens, P->B, t, &b, &p);
    int n = p + 1;
    cand* c = (cand*)malloc(sizeof(cand) * (size_t)n);
    int* sel = (int*)malloc(sizeof(int) * (size_t)(n < P->K ? n : P->K));
    if (!c || !sel) {
      free(c);
      free(sel);
#pragma omp atomic write
      err = ORC_ENOMEM;
      continue;
    }
    for (int j = 0; j < n; ++j) {
      c[j].s = li_score(P, t, b, j, NULL);
      c[j].j = j;
    }
    qsort(c, (size_t)n, sizeof(cand), by_score_then_pos);
    int m = n < P->K ? n : P->K;
    for (int r = 0; r < m; ++r) sel[r] = c[r].j;
    if (out_kth) out_kth[i] = c[m - 1].s;
    qsort(sel, (size_t)m, sizeof(int), by_int);
    int* row = out_idx + (long long)i * P->K;
    for (int r = 0; r < P->K; ++r) row[r] = r < m ? sel[r] : -1;
    if (out_cnt) out_cnt[i] = m;
    free(c);
    free(sel);
  }
  return err;
}

/* ---- Sparse Flash Attention over a given index set ----------------------------------- */

static int sfa_check(const orc_sfa* S) {
  if (!S || S->B <= 0 || S->n_q < 0 || S->H <= 0 || S->d_qk <= 0 || S->d_v <= 0 ||
      S->d_v > S->d_qk || S->K <= 0 || S->page_size <= 0 || S->max_pages <= 0 || !S->q ||
      !S->kv_pool || !S->page_table || !S->seq_lens || !S->q_start)
    return ORC_EARG;
  return ORC_OK;
}

/* out[i][h][0..d_v) and lse[i][h] for each listed token over its K indices (entries -1 are
 * skipped; any other entry must be a position < seq_len of the token's sequence). */
int oracle_sfa(const orc_sfa* S, int n_tok, const int* toks, const int* idx, double* out,
               double* lse) {
  int rc = sfa_check(S);
  if (rc) return rc;
  if (n_tok < 0 || (n_tok > 0 && (!toks || !idx || !out))) return ORC_EARG;
  for (int i = 0; i < n_tok; ++i) {
    int b, p;
    if (toks[i] < 0 || toks[i] >= S->n_q) return ORC_EARG;
    if (locate(S->q_start, S->seq_lens, S->B, toks[i], &b, &p)) return ORC_EARG;
    for (int r = 0; r < S->K; ++r) {
      int j = idx[(long long)i * S->K + r];
      if (j < -1 || j >= S->seq_lens[b]) return ORC_EINDEX;
      if (j >= 0) {
        int pg = S->page_table[(long long)b * S->max_pages + j / S->page_size];
        if (pg < 0 || pg >= S->num_pages) return ORC_EINDEX;
      }
    }
  }
  int err = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
  for (int i = 0; i < n_tok; ++i) {
    for (int h = 0; h < S->H; ++h) {
      int t = toks[i], b, p;
      locate(S->q_start, S->seq_lens, S->B, t, &b, &p);
      const int* set = idx + (long long)i * S->K;
      double* o = out + ((long long)i * S->H + h) * S->d_v;
      const uint16_t* qh = S->q + ((long long)t * S->H + h) * S->d_qk;
      double* z = (double*)malloc(sizeof(double) * (size_t)S->K);
      if (!z) {
#pragma omp atomic write
        err = ORC_ENOMEM;
        continue;
      }
      double zmax = -INFINITY;
      for (int r = 0; r < S->K; ++r) {
        int j = set[r];
        if (j < 0) continue;
        const uint16_t* kv = S->kv_pool + phys_row(S->page_table, S->max_pages, S->page_size, b, j) * S->d_qk;
        double dot = 0.0;
        for (int d = 0; d < S->d_qk; ++d) dot += orc_bf16(qh[d]) * orc_bf16(kv[d]);
        z[r] = S->scale * dot;
        if (z[r] > zmax) zmax = z[r];
      }
      for (int d = 0; d < S->d_v; ++d) o[d] = 0.0;
      double denom = 0.0;
      for (int r = 0; r < S->K; ++r) {
        int j = set[r];
        if (j < 0) continue;
        const uint16_t* kv = S->kv_pool + phys_row(S->page_table, S->max_pages, S->page_size, b, j) * S->d_qk;
        double a = exp(z[r] - zmax);
        denom += a;
        for (int d = 0; d < S->d_v; ++d) o[d] += a * orc_bf16(kv[d]);
      }
      if (denom > 0.0)
        for (int d = 0; d < S->d_v; ++d) o[d] /= denom;
      if (lse) lse[(long long)i * S->H + h] = denom > 0.0 ? zmax + log(denom) : -INFINITY;
      free(z);
    }
  }
  return err;
}

int oracle_abi_version(void) { return 2; }
