/*
 * dsa.h -- C ABI of the DSA (Dynamic Sparse Attention) hot path for GB300 (sm_103a).
 *
 * The path, as the public pages on Kimi K3.1 Pro inference describe it:
 *   1. Lightning Indexer: score the query against every cached key with per-head weights
 *      ("Inference Optimization for Kimi K3.1 Pro: Decoding Architecture Evolution and Systems
 *      Engineering Practices", section 1, DSA step 1; "Day0 Inference Adaptation for Next-Gen
 *      LLMs ... CANN", section 3.1),
 *   2. keep the top-K positions, fused with scoring so that no score reaches global memory
 *      (first page, section 2 "Operator-Level Deep Fusion"),
 *   3. Sparse Flash Attention over only those positions of the paged MLA latent cache, blockwise
 *      with a cross-block softmax reduction ("Optimizing Kimi K3.1 Pro Sparse Attention
 *      Inference ...", section "Inheritance and Extension of Core Operators").
 *
 * Conventions shared by every call:
 *   - Every pointer in an args struct is a DEVICE pointer owned by the caller.  The library never
 *     allocates, never frees, never synchronises and keeps no pointer after it returns.  Work is
 *     enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and runs
 *     asynchronously.
 *   - Synchronous errors (bad shape, null pointer, unsupported specialisation) are returned
 *     before anything is launched; dsa_last_error() then holds a one-line reason for the calling
 *     thread.  A failed launch returns DSA_ERR_CUDA.
 *   - Device-side checks (an index, length or page id out of range, a bounded wait that ran out)
 *     never trap: the kernel skips the offending work and stores a DSA_ERR_* code into *status
 *     (when status is not NULL; first error wins).  The caller reads it after synchronising.
 *   - Caches are paged with `page_size` rows per page.  Logical position j of sequence b lives at
 *     physical row page_table[b * max_pages + j / page_size] * page_size + j % page_size.
 *   - Query tokens are packed over sequences: the tokens of sequence b are q_start[b] ..
 *     q_start[b+1]-1; they are the last n_b = q_start[b+1]-q_start[b] positions of the sequence,
 *     so token i of sequence b sits at position seq_lens[b] - n_b + i (the keys and latent rows of
 *     the new tokens are already in the caches) and sees positions 0 .. that position.
 *   - Indices are LOGICAL positions, so results do not depend on where pages are placed.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 7

/* Same type as cudaStream_t. */
typedef struct CUstream_st* dsa_stream_t;

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,  /* null pointer, negative or inconsistent size                    */
  DSA_ERR_UNSUPPORTED = 2,  /* valid, but no compiled specialisation covers it                */
  DSA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or a launch failed                  */
  DSA_ERR_DEVICE_CHECK = 4, /* (in *status) a device-side range check failed                  */
  DSA_ERR_TIMEOUT = 5       /* (in *status) a bounded device-side wait gave up                */
} dsa_status;

/* DSA_MXFP8_E4M3: e4m3 elements with one E8M0 (power-of-two) scale per 32 consecutive elements. */
typedef enum { DSA_BF16 = 0, DSA_FP8_E4M3 = 1, DSA_MXFP8_E4M3 = 2 } dsa_dtype;

/* Human-readable name of a status code (static storage). */
const char* dsa_status_string(dsa_status s);

/* Reason for the last synchronous error returned on the calling thread ("" if none). */
const char* dsa_last_error(void);

/* DSA_ABI_VERSION of the built library. */
int dsa_abi_version(void);

/* ------------------------------------------------------------------------------------------ */
/* Lightning Indexer + top-K                                                                   */
/* ------------------------------------------------------------------------------------------ */

/*
 * For every query token t (at position p):
 *   s(t, j) = sum_{h < H_I} w[t][h] * max(0, q[t][h][:] . k[j][:])      for 0 <= j <= p,
 * with one index key row k[j] (d_I wide) per position, shared by all index heads; in FP8 mode
 * q[t][h][:] = q8 * q_scale[t][h] and k[j][:] = k8 * k_scale[row(j)]; in MXFP8 mode
 * ("Inference Optimization for Kimi K3.1 Pro", section 4: the indexer's fully quantised path,
 * group size 32) q[t][h][d] = q8 * 2^(q_sf[t][h][d/32] - 127) and
 * k[j][d] = k8 * 2^(k_sf[row(j)][d/32] - 127) (E8M0 bytes; 255 is not a valid scale).  The
 * selected set is the
 * first min(K, p+1) positions in the order (score descending, position ascending) -- ties go to
 * the lower position, and -0.0 equals +0.0.  Scores never leave the chip.
 *
 * Supported: page_size 64; (H_I, d_I) in {(8, 64), (64, 128)}; dtype BF16, or FP8_E4M3 and
 * MXFP8_E4M3 with (H_I, d_I) = (64, 128);
 * 1 <= K <= 2048; max_seq_len <= 131072; any number of tokens per sequence (decode, speculative
 * multi-token decode, chunked prefill).
 *
 * Position units (decode and two-token groups, max_seq_len > 32768, B <= 256): a sequence longer than one
 * cluster's span (32768 positions) is split into equal units, each selecting the top-K of its own
 * positions (with their scores) into `workspace`; a second kernel then merges each such token's
 * units ("Inference Optimization for Kimi K3.1 Pro", section 5: a local Top-K before the
 * merge, here over ranges of one sequence on one GPU), so that a batch of short and long
 * sequences spreads evenly over the SMs.  The result is the same set, in the same order.
 * dsa_li_workspace_bytes() says how much scratch that takes (0 when no sequence can be split).
 */
typedef struct {
  int B;            /* sequences                                                         */
  int n_q;          /* query tokens over all sequences (= q_start[B])                    */
  int H_I, d_I;     /* index heads, index head dim                                        */
  int K;            /* top-K                                                              */
  int page_size;    /* rows per page (64)                                                 */
  int max_pages;    /* row stride of page_table                                           */
  int num_pages;    /* pages in k_pool (device check on every page id)                     */
  int max_seq_len;  /* host-known upper bound of seq_lens[] (sizes the launch)            */
  int max_q_per_seq;/* host-known upper bound of q_start[b+1]-q_start[b]                  */
  dsa_dtype dtype;
  const void* q;          /* [n_q][H_I][d_I]   bf16 | e4m3                                */
  const float* q_scale;   /* [n_q][H_I] fp32, FP8 only (per-token scales: replicate)      */
  const float* w;         /* [n_q][H_I] fp32 head weights                                 */
  const void* k_pool;     /* [num_pages][page_size][d_I]  bf16 | e4m3                     */
  const float* k_scale;   /* [num_pages][page_size] fp32, FP8 only                        */
  const int32_t* page_table; /* [B][max_pages] physical page ids                          */
  const int32_t* seq_lens;   /* [B] positions, new tokens included                        */
  const int32_t* q_start;    /* [B+1] prefix offsets of the query tokens                  */
  int32_t* out_idx;       /* [n_q][K] selected positions, ascending, then -1 padding      */
  int32_t* out_cnt;       /* [n_q] number selected = min(K, p+1), or NULL                 */
  int32_t* status;        /* device int32 error word, or NULL                             */
  const uint8_t* q_sf;    /* [n_q][H_I][d_I/32] E8M0 group scales, MXFP8 only (else NULL) */
  const uint8_t* k_sf;    /* [num_pages][page_size][d_I/32] E8M0, MXFP8 only; the 4-byte
                             row of scales must be 4-byte aligned (d_I = 128)              */
  float* out_score;       /* [n_q][K] fp32 score of each position in out_idx (-inf for the
                             padding), or NULL: the candidates of a context-parallel shard  */
  void* workspace;        /* device scratch of dsa_li_workspace_bytes() bytes, 256-B aligned,
                             or NULL when that is 0; owned by the caller, no initial value */
  size_t workspace_bytes;
} dsa_li_args;

/* Scratch that dsa_li_topk needs for these arguments (0 if none).  Host only: reads B, K,
 * max_seq_len and max_q_per_seq; no CUDA call. */
size_t dsa_li_workspace_bytes(const dsa_li_args* args);

dsa_status dsa_li_topk(const dsa_li_args* args, dsa_stream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* Sparse Flash Attention                                                                      */
/* ------------------------------------------------------------------------------------------ */

/*
 * For every query token t and head h, over the index set S_t = {idx[t][r] : idx[t][r] >= 0}:
 *   z_j = softmax_scale * q[t][h][0:d_qk] . kv[j][0:d_qk]
 *   out[t][h][:] = sum_j exp(z_j - m) kv[j][0:d_v] / sum_j exp(z_j - m),   m = max_j z_j
 *   lse[t][h]    = m + ln(sum_j exp(z_j - m))
 * The value is the leading d_v columns of the same latent row (MLA), so each selected row is
 * read once.  An empty set gives out = 0 and lse = -inf.  An index >= seq_lens[b] or < -1 is a
 * device check failure: the row is skipped and *status set.
 *
 * dsa_sfa_decode targets few tokens per sequence: it splits each token's K rows over several CTA
 * pairs and merges the partial softmax states through `workspace` (dsa_sfa_workspace_bytes()
 * bytes; with two splits, the usual case, each split finalises half of the heads);
 * dsa_sfa_prefill targets many tokens per sequence (one token per CTA pair, no workspace).  Both
 * give the same result up to fp32 rounding.
 *
 * Stream order: both are launched as programmatic dependents of the preceding kernel in the
 * stream, so their CTAs may start (barrier set-up, tensor-memory allocation) while that kernel
 * finishes; they read no device memory (inputs included) before it has completed.  Stream order
 * is therefore kept for every input, whichever kernel wrote it.
 *
 * Supported: page_size 64; d_qk 576; d_v 512; H in {16, 128} (decode) and 128 (prefill);
 * 1 <= K <= 2048; bf16 q/out; latent cache bf16 or FP8 (kv_dtype).
 *
 * FP8 latent cache (kv_dtype DSA_FP8_E4M3; "Inference Optimization for Kimi K3.1 Pro",
 * section 4, SFA KV cache quantisation per token and 128-column tile): each row of kv_pool is
 * 608 bytes: the 576 columns as e4m3 codes, then one fp32 scale per 128-column tile (5; the
 * last covers the 64 rope columns), then 12 unused bytes.  The attention runs on the BF16
 * values bf16(fp32(code * scale)) (both roundings to nearest even).
 */
typedef struct {
  int B, n_q;
  int H;              /* query heads                                                     */
  int d_qk, d_v;      /* 576, 512                                                        */
  int K;              /* row stride of idx                                               */
  int page_size, max_pages, num_pages;
  int max_seq_len, max_q_per_seq;
  float softmax_scale;
  const void* q;             /* [n_q][H][d_qk] bf16                                      */
  const void* kv_pool;       /* [num_pages][page_size][d_qk] bf16                        */
  const int32_t* page_table; /* [B][max_pages]                                           */
  const int32_t* seq_lens;   /* [B]                                                      */
  const int32_t* q_start;    /* [B+1]                                                    */
  const int32_t* idx;        /* [n_q][K] logical positions, -1 = empty slot              */
  void* out;                 /* [n_q][H][d_v] bf16                                       */
  float* lse;                /* [n_q][H] fp32, or NULL                                   */
  int32_t* status;           /* device int32 error word, or NULL                         */
  void* workspace;           /* device scratch of dsa_sfa_workspace_bytes(), 256-B aligned */
  size_t workspace_bytes;
  dsa_dtype kv_dtype;        /* DSA_BF16 (rows of 576 bf16) or DSA_FP8_E4M3 (608-byte rows) */
  int row_splits;            /* dsa_sfa_decode: CTA pairs that share one token's K rows
                                (0 = chosen from the SM count; the result does not depend on
                                it beyond fp32 rounding); ignored by dsa_sfa_prefill        */
} dsa_sfa_args;

/* Scratch that dsa_sfa_decode needs for these arguments (0 if none).  Host only: it reads the
 * current device's SM count (the split plan depends on it; 152 when no device is visible) and
 * launches nothing.  Only n_q, H, K and row_splits are read. */
size_t dsa_sfa_workspace_bytes(const dsa_sfa_args* args);

dsa_status dsa_sfa_decode(const dsa_sfa_args* args, dsa_stream_t stream);
dsa_status dsa_sfa_prefill(const dsa_sfa_args* args, dsa_stream_t stream);

/*
 * dsa_sfa_decode without a caller workspace, for callers that cannot allocate device memory: an
 * operator inside a framework that plans all device memory itself and passes the operator only
 * its inputs and outputs, or a path on which allocating is not allowed.  The pages have no
 * counterpart of this; it is an interface convenience of this library.
 *
 * The split-merge scratch is a fixed device array of DSA_SFA_STATIC_SCRATCH_BYTES inside the
 * library, held by every GPU that loads the library until the process exits.  args->workspace and
 * args->workspace_bytes are ignored; everything else is exactly dsa_sfa_decode (same kernel, same
 * result).  Arguments whose dsa_sfa_workspace_bytes() exceeds the capacity are rejected with
 * DSA_ERR_UNSUPPORTED and a reason in dsa_last_error().  No call allocates or frees memory.
 *  - The first call on a device looks up the array's device address (once per device, with that
 *    device current); make that first call before capturing a stream.
 *  - All calls on a device share the one array, which keeps the last call's contents; the call
 *    clears what must start at zero.  Calls whose work overlaps on the GPU (other streams, other
 *    host threads) race on the array: serialise them.
 *  - Capacity: with row_splits = 0 and K <= 2048 the library never plans more CTA pairs than
 *    one wave holds (2 * n_q * splits <= SMs), and a plan needs at most
 *    n_q * splits * 263,168 bytes (+ 512 for alignment and counters), so 20 MiB covers every such
 *    plan on a GPU of 159 SMs or fewer (152 on GB300).  An explicit row_splits or a larger K can
 *    exceed it; such calls are rejected as above.
 */
#define DSA_SFA_STATIC_SCRATCH_BYTES (20u * 1024u * 1024u)
dsa_status dsa_sfa_decode_static(const dsa_sfa_args* args, dsa_stream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* Context-parallel top-K merge                                                                */
/* ------------------------------------------------------------------------------------------ */

/*
 * "Inference Optimization for Kimi K3.1 Pro", section 5 (local Top-K before communication): a
 * long sequence's positions are split over S shards; each shard runs dsa_li_topk on its own
 * range (with out_score) and the shards' (score, position) candidates are gathered -- the one
 * exchange step -- and merged here.  For each query t the result is the first min(K, valid)
 * candidates in the order (score descending, position ascending), emitted in ascending
 * position order with -1 padding: the same set dsa_li_topk selects over the whole range, since
 * every position's score does not depend on the split.
 *   cand_idx   [S][n_q][K_in] shard-local positions (-1 = none); position + shard_offset[s] is
 *              the sequence position (shards own disjoint ranges)
 *   cand_score [S][n_q][K_in] their scores
 * Supported: S * K_in <= 16384, K <= K_in * S.  Device pointers; asynchronous on stream.
 */
typedef struct {
  int S, n_q, K_in, K;
  const int32_t* cand_idx;
  const float* cand_score;
  const int32_t* shard_offset; /* [S] device array                                          */
  int32_t* out_idx;            /* [n_q][K]                                                   */
  int32_t* out_cnt;            /* [n_q] or NULL                                              */
} dsa_topk_merge_args;

dsa_status dsa_topk_merge(const dsa_topk_merge_args* args, dsa_stream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* Indexer Prolog                                                                              */
/* ------------------------------------------------------------------------------------------ */

/*
 * The indexer's input preparation for the new tokens ("Inference Optimization for Kimi K3.1 Pro",
 * section 3, Indexer Prolog, and section 4, MXFP8 indexer path; "Day0 Inference Adaptation ...
 * CANN", section 3.3).  For each new token t (sequence b, position p = seq_lens[b] - n_b + i):
 *   q[t][h][:] = W_q[h*d_I .. h*d_I+d_I) . xq[t]                 -> q_out (+ q_sf)
 *   k[t]       = LayerNorm(W_k . x[t]) * ln_gamma + ln_beta        -> key-cache row of p
 *   w[t][h]    = w_scale * (W_w[h] . x[t])                         -> w_out (fp32)
 * LayerNorm: mean and biased variance over the d_I features, then (v - mean) / sqrt(var + eps).
 * dtype DSA_MXFP8_E4M3: q and k become e4m3 codes with one E8M0 scale byte per 32 features
 * (shared exponent floor(log2(max |v|)) - 8, clamped to [-127, 127], 0 for an all-zero group;
 * elements v / 2^e rounded to nearest even, saturated at 448; a zero is +0) -- the layout
 * dsa_li_topk reads in its MXFP8 mode; dtype DSA_BF16: bf16, round to nearest even.
 * The three projections run as concurrent CTA roles of one launch (no stream fork).
 *
 * Supported: H_I = 64, d_I = 128, page_size 64; d_q and d_model multiples of 8; bf16 inputs and
 * weights, 16-byte aligned.  A position whose page id is outside [0, num_pages) sets
 * DSA_ERR_DEVICE_CHECK and its key row is not written.
 */
typedef struct {
  int n_q;              /* new tokens (= q_start[B])                                       */
  int B;
  int d_q;              /* input width of the Q projection                                 */
  int d_model;          /* input width of the K and head-weight projections                */
  int H_I, d_I;         /* 64, 128                                                         */
  dsa_dtype dtype;      /* DSA_MXFP8_E4M3 or DSA_BF16: format of q_out and of the key cache */
  int page_size;        /* 64                                                              */
  int max_pages;        /* row stride of page_table                                        */
  int num_pages;        /* pages in k_pool                                                 */
  float ln_eps;
  float w_scale;        /* head-weight scale                                               */
  const void* xq;       /* [n_q][d_q] bf16                                                 */
  const void* x;        /* [n_q][d_model] bf16                                             */
  const void* w_q;      /* [H_I*d_I][d_q] bf16                                             */
  const void* w_k;      /* [d_I][d_model] bf16                                             */
  const void* w_w;      /* [H_I][d_model] bf16                                             */
  const float* ln_gamma;/* [d_I]                                                           */
  const float* ln_beta; /* [d_I]                                                           */
  const int32_t* page_table; /* [B][max_pages] of the key cache                           */
  const int32_t* seq_lens;   /* [B] positions, new tokens included                        */
  const int32_t* q_start;    /* [B+1]                                                     */
  void* q_out;          /* [n_q][H_I][d_I] e4m3 codes or bf16                              */
  uint8_t* q_sf;        /* [n_q][H_I][d_I/32] (MXFP8)                                      */
  float* w_out;         /* [n_q][H_I]                                                      */
  void* k_pool;         /* [num_pages][page_size][d_I] e4m3 codes or bf16 (written rows only) */
  uint8_t* k_sf;        /* [num_pages][page_size][d_I/32] (MXFP8)                          */
  void* workspace;      /* unused: dsa_prolog_workspace_bytes() is 0 (the slices of a tile
                           meet in distributed shared memory); may be NULL                */
  size_t workspace_bytes;
  int32_t* status;      /* device int32 error word, or NULL                                */
} dsa_prolog_args;

/* Scratch bytes dsa_indexer_prolog needs for these sizes (only the size fields are read): 0 --
 * this implementation needs none; kept so that callers size the field the same way as the
 * other entry points' workspaces. */
size_t dsa_prolog_workspace_bytes(const dsa_prolog_args* args);
dsa_status dsa_indexer_prolog(const dsa_prolog_args* args, dsa_stream_t stream);

/* ------------------------------------------------------------------------------------------ */
/* Cache layout and page-table helpers                                                         */
/* ------------------------------------------------------------------------------------------ */

/*
 * The caches are paged: the indexer reads the paged key cache directly ("Day0 Inference
 * Adaptation for Next-Gen LLMs ... CANN", section 3.1), and the selected indices address the
 * paged KV cache page by page ("Inference Optimization for Kimi K3.1 Pro", section 2, "Inlined
 * Top-K Selection": on-demand in-page addressing).  The helpers below describe and maintain
 * that layout; they are host-side conveniences (the pages define no interface).
 */

/* Bytes of one page of `rows` rows of `dim` elements of `dtype` (0 on invalid input); for
 * MXFP8 the elements only (the E8M0 scales are a separate [rows][dim/32] byte array, the
 * group-32 scales of "Inference Optimization for Kimi K3.1 Pro", section 4). */
size_t dsa_page_bytes(dsa_dtype dtype, int rows, int dim);

/*
 * Host-side check of a page table (host pointers) before it drives the in-page addressing of
 * the kernels ("Inference Optimization for Kimi K3.1 Pro", section 2, "Inlined Top-K
 * Selection"): for every sequence b, the pages
 * 0 .. ceil(seq_lens[b]/page_size)-1 hold ids in [0, num_pages), and (if require_unique) no id
 * is used twice over the whole table.  Entries past a sequence's last page are ignored.
 * Returns DSA_OK or DSA_ERR_INVALID_ARG (reason in dsa_last_error()).
 */
dsa_status dsa_page_table_validate(const int32_t* page_table_host, int B, int max_pages,
                                   const int32_t* seq_lens_host, int page_size, int num_pages,
                                   int require_unique);

/*
 * Append new rows to a paged cache: the write of the new tokens' keys that the indexer's input
 * preparation performs ("Inference Optimization for Kimi K3.1 Pro", section 3, "Three-Stream
 * Parallel Architecture", the K normalisation stream; dsa_indexer_prolog does this itself for
 * the key cache), or of latent rows for the attention cache.  Scatter n_rows rows (device
 * pointers):
 *   pool[page_table[seq[r]][pos[r] / page_size]][pos[r] % page_size][:] = rows[r][:]
 * and, when row_scales is not NULL, scale_pool[same page][same slot] = row_scales[r] (the
 * per-row fp32 scale of an FP8 key cache).  elem_bytes is 2 (bf16) or 1 (e4m3); dim*elem_bytes
 * must be a multiple of 16.  Out-of-range seq/pos/page entries are skipped and flagged in
 * *status.
 */
dsa_status dsa_cache_write(void* pool, float* scale_pool, int num_pages, int page_size, int dim,
                           int elem_bytes, const int32_t* page_table, int max_pages, int B,
                           const int32_t* seq, const int32_t* pos, const void* rows,
                           const float* row_scales, int n_rows, int32_t* status,
                           dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
