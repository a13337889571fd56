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
 *              o = 0 and lse = -inf.  With an FP8 latent cache kv[j,d] is the de-quantised
 *              bf16(fp32(e4m3 code * tile scale)), one fp32 scale per row and 128 columns.
 *   prolog     projections, LayerNorm and OCP MX quantisation of the indexer's inputs (see
 *              the Indexer Prolog section below).
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
  int kv_fp8;                 /* 1: the latent cache is FP8 rows (kv8_pool), else bf16    */
  const uint8_t* kv8_pool;    /* [num_pages][page_size][608]: 576 e4m3 codes, then one
                                 fp32 scale per 128-column tile (5; the last tile is the 64
                                 rope columns), then 12 bytes of padding                   */
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

static uint16_t orc_bf16_encode(double v);

/* FP8 latent cache ("Inference Optimization for Kimi K3.1 Pro", section 4, SFA KV cache
 * quantisation: the cache is stored in FP8 with one scale per token and 128-column tile, and
 * the attention arithmetic runs on the de-quantised BF16 values).  Element d of a row is the
 * e4m3 code times its tile's fp32 scale, the product rounded to fp32 and then to bf16 (the
 * precision in which a BF16 tensor-core operand is formed from the stored pair). */
#define ORC_KV8_ROW 608
double orc_kv8_element(const uint8_t* row, int d) {
  float sc;
  memcpy(&sc, row + 576 + 4 * (d / 128), sizeof sc);
  const float prod = (float)orc_e4m3(row[d]) * sc;
  return orc_bf16(orc_bf16_encode((double)prod));
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
      !(S->kv_fp8 ? (const void*)S->kv8_pool : (const void*)S->kv_pool) || !S->page_table ||
      !S->seq_lens || !S->q_start)
    return ORC_EARG;
  if (S->kv_fp8 && S->d_qk != 576) return ORC_EARG;
  return ORC_OK;
}

/* Element d of the latent row at physical row `row` (bf16 cache, or de-quantised FP8 row). */
static double sfa_kv(const orc_sfa* S, long long row, int d) {
  if (S->kv_fp8) return orc_kv8_element(S->kv8_pool + row * ORC_KV8_ROW, d);
  return orc_bf16(S->kv_pool[row * S->d_qk + d]);
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
        const long long row = phys_row(S->page_table, S->max_pages, S->page_size, b, j);
        double dot = 0.0;
        for (int d = 0; d < S->d_qk; ++d) dot += orc_bf16(qh[d]) * sfa_kv(S, row, d);
        z[r] = S->scale * dot;
        if (z[r] > zmax) zmax = z[r];
      }
      for (int d = 0; d < S->d_v; ++d) o[d] = 0.0;
      double denom = 0.0;
      for (int r = 0; r < S->K; ++r) {
        int j = set[r];
        if (j < 0) continue;
        const long long row = phys_row(S->page_table, S->max_pages, S->page_size, b, j);
        double a = exp(z[r] - zmax);
        denom += a;
        for (int d = 0; d < S->d_v; ++d) o[d] += a * sfa_kv(S, row, d);
      }
      if (denom > 0.0)
        for (int d = 0; d < S->d_v; ++d) o[d] /= denom;
      if (lse) lse[(long long)i * S->H + h] = denom > 0.0 ? zmax + log(denom) : -INFINITY;
      free(z);
    }
  }
  return err;
}

/* ---- Indexer Prolog: the indexer's input preparation -------------------------------- */
/*
 * "Inference Optimization for Kimi K3.1 Pro", section 3 (Indexer Prolog) and section 5
 * (three-stream prolog); "Day0 Inference Adaptation ... CANN", section 3.3 (the indexer fully
 * quantised to MXFP8 with group size 32, projections kept in BF16).  For each new token t:
 *   Q projection      q[t]   = W_q . xq[t]                 ([H_I*d_I], row f = h*d_I + d)
 *   K normalisation   k[t]   = LayerNorm(W_k . x[t]) * gamma + beta   (over the d_I features)
 *   head weights      w[t]   = w_scale * (W_w . x[t])       ([H_I])
 *   quantisation      q[t] and k[t] to MXFP8 (OCP Microscaling rule, groups of 32 features) or
 *                     to bf16 (round to nearest even); k[t] is written to the key cache at the
 *                     token's position p_t: row pt[b][p_t / page_size] * page_size + p_t % page_size.
 */

/* Nearest e4m3 code to y (|y| clamped to 448 first), ties to the even code; from the format's
 * value table (orc_e4m3), searched exhaustively. */
static uint8_t orc_e4m3_encode(double y) {
  int neg = y < 0.0;
  double a = fabs(y);
  if (a > 448.0) a = 448.0;
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c < 127; ++c) { /* 0x00 .. 0x7E: every finite non-negative code */
    double d = fabs(orc_e4m3((uint8_t)c) - a);
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  if (best == 0) return 0; /* +0 (a signed zero carries no information here) */
  return (uint8_t)(best | (neg ? 0x80 : 0));
}

/* bf16 bits nearest to v: 8 significant bits, ties to even (rint in the default rounding mode),
 * for v in bf16's normal range. */
static uint16_t orc_bf16_encode(double v) {
  if (v == 0.0) return signbit(v) ? 0x8000 : 0;
  int e;
  double m = frexp(v, &e);                   /* |m| in [0.5, 1) */
  float f = (float)ldexp(rint(ldexp(m, 8)), e - 8); /* exactly representable */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

/* OCP Microscaling quantisation of n values (n a multiple of 32), group by group: shared exponent
 * e = floor(log2(amax)) - 8 (8 = exponent of e4m3's largest normal), clamped to [-127, 127], 0 for
 * an all-zero group; scale byte e + 127; codes = nearest e4m3 to v / 2^e. */
int oracle_mx_quantize(const double* v, int n, uint8_t* codes, uint8_t* sf) {
  if (!v || !codes || !sf || n < 0 || n % 32) return ORC_EARG;
  for (int g = 0; g < n / 32; ++g) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i)
      if (fabs(v[g * 32 + i]) > amax) amax = fabs(v[g * 32 + i]);
    int e = 0;
    if (amax > 0.0) {
      int ex;
      frexp(amax, &ex); /* amax = m * 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1 */
      e = ex - 1 - 8;
      if (e < -127) e = -127;
      if (e > 127) e = 127;
    }
    sf[g] = (uint8_t)(e + 127);
    for (int i = 0; i < 32; ++i) codes[g * 32 + i] = orc_e4m3_encode(ldexp(v[g * 32 + i], -e));
  }
  return ORC_OK;
}

typedef struct {
  int n_q, B, d_q, d_model, H_I, d_I;
  int mx;                     /* 1: MXFP8 outputs; 0: bf16 outputs                     */
  const uint16_t* xq;         /* [n_q][d_q] bf16, input of the Q projection              */
  const uint16_t* x;          /* [n_q][d_model] bf16, input of the K and weight projections */
  const uint16_t* w_q;        /* [H_I*d_I][d_q] bf16                                     */
  const uint16_t* w_k;        /* [d_I][d_model] bf16                                     */
  const uint16_t* w_w;        /* [H_I][d_model] bf16                                     */
  const float* ln_gamma;      /* [d_I]                                                   */
  const float* ln_beta;       /* [d_I]                                                   */
  double ln_eps, w_scale;
  const int* page_table;      /* [B][max_pages]                                          */
  int max_pages, page_size;
  const int* seq_lens;        /* [B]                                                     */
  const int* q_start;         /* [B+1]                                                   */
} orc_prolog;

/* Fills, per token: q_val [n_q][H_I*d_I] and k_val [n_q][d_I] (fp64, before rounding),
 * w_out [n_q][H_I]; the encoded q (q_enc: e4m3 codes or bf16 bits, q_sf) and k (k_enc, k_sf);
 * k_row [n_q] = physical key-cache row of the token.  Any output pointer may be NULL. */
int oracle_prolog(const orc_prolog* P, double* q_val, double* k_val, double* w_out, void* q_enc,
                  uint8_t* q_sf, void* k_enc, uint8_t* k_sf, long long* k_row) {
  if (!P || P->n_q < 0 || P->B <= 0 || P->d_q <= 0 || P->d_model <= 0 || P->H_I <= 0 ||
      P->d_I <= 0 || P->d_I % 32 || !P->xq || !P->x || !P->w_q || !P->w_k || !P->w_w ||
      !P->ln_gamma || !P->ln_beta || !P->page_table || !P->seq_lens || !P->q_start ||
      P->page_size <= 0)
    return ORC_EARG;
  const int F = P->H_I * P->d_I;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < P->n_q; ++t) {
    double* q = (double*)malloc(sizeof(double) * (size_t)F);
    double* k = (double*)malloc(sizeof(double) * (size_t)P->d_I);
    uint8_t* c = (uint8_t*)malloc((size_t)F);
    uint8_t* g = (uint8_t*)malloc((size_t)F / 32);
    if (!q || !k || !c || !g) {
      free(q); free(k); free(c); free(g);
#pragma omp atomic write
      err = ORC_ENOMEM;
      continue;
    }
    for (int f = 0; f < F; ++f) {
      double acc = 0.0;
      for (int i = 0; i < P->d_q; ++i)
        acc += orc_bf16(P->w_q[(long long)f * P->d_q + i]) * orc_bf16(P->xq[(long long)t * P->d_q + i]);
      q[f] = acc;
    }
    for (int d = 0; d < P->d_I; ++d) {
      double acc = 0.0;
      for (int i = 0; i < P->d_model; ++i)
        acc += orc_bf16(P->w_k[(long long)d * P->d_model + i]) * orc_bf16(P->x[(long long)t * P->d_model + i]);
      k[d] = acc;
    }
    double mean = 0.0, var = 0.0;
    for (int d = 0; d < P->d_I; ++d) mean += k[d];
    mean /= P->d_I;
    for (int d = 0; d < P->d_I; ++d) var += (k[d] - mean) * (k[d] - mean);
    var /= P->d_I;
    const double rstd = 1.0 / sqrt(var + P->ln_eps);
    for (int d = 0; d < P->d_I; ++d)
      k[d] = (k[d] - mean) * rstd * (double)P->ln_gamma[d] + (double)P->ln_beta[d];
    if (w_out)
      for (int h = 0; h < P->H_I; ++h) {
        double acc = 0.0;
        for (int i = 0; i < P->d_model; ++i)
          acc += orc_bf16(P->w_w[(long long)h * P->d_model + i]) * orc_bf16(P->x[(long long)t * P->d_model + i]);
        w_out[(long long)t * P->H_I + h] = P->w_scale * acc;
      }
    if (q_val) memcpy(q_val + (long long)t * F, q, sizeof(double) * (size_t)F);
    if (k_val) memcpy(k_val + (long long)t * P->d_I, k, sizeof(double) * (size_t)P->d_I);
    if (P->mx) {
      oracle_mx_quantize(q, F, c, g);
      if (q_enc) memcpy((uint8_t*)q_enc + (long long)t * F, c, (size_t)F);
      if (q_sf) memcpy(q_sf + (long long)t * F / 32, g, (size_t)F / 32);
      oracle_mx_quantize(k, P->d_I, c, g);
      if (k_enc) memcpy((uint8_t*)k_enc + (long long)t * P->d_I, c, (size_t)P->d_I);
      if (k_sf) memcpy(k_sf + (long long)t * P->d_I / 32, g, (size_t)P->d_I / 32);
    } else {
      if (q_enc)
        for (int f = 0; f < F; ++f) ((uint16_t*)q_enc)[(long long)t * F + f] = orc_bf16_encode(q[f]);
      if (k_enc)
        for (int d = 0; d < P->d_I; ++d)
          ((uint16_t*)k_enc)[(long long)t * P->d_I + d] = orc_bf16_encode(k[d]);
    }
    if (k_row) {
      int b, p;
      if (locate(P->q_start, P->seq_lens, P->B, t, &b, &p) ||
          p / P->page_size >= P->max_pages) {
        k_row[t] = -1;
      } else {
        k_row[t] = phys_row(P->page_table, P->max_pages, P->page_size, b, p);
      }
    }
    free(q); free(k); free(c); free(g);
  }
  return err;
}

int oracle_abi_version(void) { return 3; }
