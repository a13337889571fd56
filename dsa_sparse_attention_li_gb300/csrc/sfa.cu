// sfa.cu -- Sparse Flash Attention over the positions chosen by the indexer, reading the paged
// MLA latent cache (576 = 512 latent + 64 rope; the value is the leading 512 columns of the same
// row) straight through the page table, with tcgen05 tensor cores for Q.K^T and P.V and an
// online softmax in between.
//
// Method: "Optimizing Kimi K3.1 Pro Sparse Attention Inference: Day0 Adaptation and Performance
// Tuning on Ascend", section "Inheritance and Extension of Core Operators" (SFA reuses
// FlashAttention's blockwise scheme: exact attention inside blocks, a careful reduction across
// blocks, no global softmax); "Inference Optimization for Kimi K3.1 Pro ...", section 2 (the
// selected indices address the paged KV cache directly, page by page, instead of contiguous
// blocks); "Day0 Inference Adaptation ... CANN", section 3.1 (SFA reads the main attention KV at
// the indexer's positions).
//
// Work decomposition.  A pair of CTAs (16 warps each) serves one (query token t, row split s);
// CTA r of the pair owns the value columns [256r, 256r + 256) and, for Q.K^T, the head
// dimensions D_r = [256r, 256r + 256) + [512 + 32r, 512 + 32r + 32) (half of the 576):
//   - Q[t] on D_r: the 256 value dimensions live in TMEM (A operand of 16 k-steps), the 32 rope
//     dimensions in shared memory (64-byte swizzle, A operand of 2 k-steps);
//   - the split's selected positions are translated to physical rows (page table) in shared
//     memory; seven gather warps copy, per 64-row tile, only the 576 bytes of each row the CTA
//     uses (its 512 value bytes and 64 rope bytes) with 16-byte cp.async (empty slots are
//     zero-filled) into a 4-stage ring (value boxes [box][row][128 B] with the 128-byte swizzle,
//     rope box with 64-byte rows), so a stage is the K-major B operand of Q.K^T (N = 64 rows)
//     and its value boxes the MN-major B operand of P.V (K = 64 rows, N = 256);
//   - S_r = Q[:, D_r].K[:, D_r]^T goes to one of two TMEM buffers.  The pair splits each tile's
//     columns for the softmax: CTA r finalises columns [32r, 32r + 32) for all 128 heads, so
//     the exponentials of every head row spread over the four TMEM lane quadrants (each served
//     by its own SM sub-partition).  Eight score warps form two teams that take alternate
//     tiles, one thread per head row: a thread sends the CTA's partial of the peer's columns
//     to the peer through distributed shared memory (asynchronous stores counted on the peer's
//     mbarrier), adds the peer's partial of its own columns (always S_0 + S_1), masks and
//     scales them, exchanges its row maximum with the peer (512 bytes a tile; both CTAs then
//     hold the same maximum and take the same rescale decisions), takes the reference maximum
//     the other team left after the previous tile, exponentiates and writes its columns of P
//     (bf16) into its P buffer and the peer's (the A operand of P.V in both).  Distributed
//     shared memory moves about 20 bytes per clock, so the tile moves 16 KiB of partial scores
//     and 8 KiB of P each way instead of both full partials (32 KiB); and with two teams one
//     tile's round trips to the peer overlap the next tile's.  The reference maximum only
//     moves when a tile's maximum exceeds it by more than 2^8; then each CTA rescales its O
//     rows;
//   - O (128 x 256 fp32 = half of TMEM) accumulates P.V_r across tiles.
// Each head's 128x512 fp32 O would fill all of TMEM, hence the value split over the pair; the
// split of the Q.K^T dimensions halves both the gathered bytes and the tensor work of each CTA.
// With two row splits both pairs of a token form one cluster of four: split s finalises heads
// [64s, 64s + 64) of its value half, the other split writes its normalised rows of those heads
// and their lse to the caller's workspace (L2) before the cluster barrier, and split s combines
// them with its own after it.  With more splits the partial (o, lse) go to the workspace and the
// last CTA of a (token, r) to finish merges them.
//
// FP8 latent cache ("Inference Optimization for Kimi K3.1 Pro", section 4: the cache stored in
// FP8 per token and 128-column tile, the attention arithmetic in BF16): rows of 576 e4m3 codes
// and 5 fp32 tile scales; the gather threads copy the codes and scales they need into the upper
// part of the tile's stage with cp.async, and convert a tile (fp32 product, bf16 rounding) into
// the same swizzled BF16 tile once the next tile's copies are issued, so everything after the
// gather is unchanged (template parameter KV8).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace sfa {

constexpr int kThreads = 512;  // 16 warps: 0-3, 9-11 gather; 8 MMA; 4-7 and 12-15 score warps
constexpr int kGatherThreads = 224;
constexpr int kMmaWarp = 8;
constexpr int kHeads = 128;        // MMA M (heads are padded to 128)
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kDvHalf = 256;
constexpr int kNT = 64;            // gathered rows per tile (MMA N of Q.K^T)
constexpr int kStages = 4;
constexpr int kBoxBytes = kNT * 128;                        // one value box of a tile: 8 KiB
constexpr int kRopeHalf = 32;      // rope columns of this CTA's half of Q.K^T
constexpr int kRopeBoxBytes = kNT * kRopeHalf * 2;          // 64-byte rows: 4 KiB
constexpr int kTileBytes = 4 * kBoxBytes + kRopeBoxBytes;   // 36 KiB
constexpr int kRowChunks = 32 + 4;                          // 16-byte chunks gathered per row
constexpr int kChunks = kNT * kRowChunks;                   // per tile (2304)
constexpr int kMaxRows = 2048;     // row slots per CTA
constexpr float kRescaleLog2 = 8.0f;
constexpr int kFinCols = kNT / 2;  // columns of a tile whose softmax this CTA finalises
// bytes that arrive per tile through distributed shared memory
constexpr uint32_t kXBytes = kHeads * kFinCols * 4;         // the peer's partial S of our columns
constexpr uint32_t kMxBytes = kHeads * 4;                   // the peer's row maxima of its columns
constexpr uint32_t kPRemBytes = kHeads * kFinCols * 2;      // the peer's columns of P (bf16)
constexpr uint32_t kFinBytes = kHeads * 8;                  // the peer's partial row sums
// TMEM columns (512 in total)
constexpr uint32_t kColQ = 0;      // Q value columns of D_r: 256 bf16 per lane = 128 columns
constexpr uint32_t kColS = 128;    // partial S, two buffers of 64 columns (tile i uses i & 1)
constexpr uint32_t kColO = 256;    // O half: 256 columns
constexpr uint32_t kTmemCols = 512;
constexpr int kGatherPer = (kChunks + kGatherThreads - 1) / kGatherThreads;  // chunks per thread
static_assert(kColQ + 128 <= kColS && kColS + 2 * kNT <= kColO, "TMEM columns");

struct Params {
  int B, n_q, H, K, max_pages, num_pages;
  int splits;      // row splits per token
  int rows_per;    // row slots per split (multiple of kNT)
  int cluster_merge;  // splits == 2: the two splits of a token share a cluster of 4 and each
                      // finalises half of the heads (rows exchanged through the workspace)
  float scale_log2;  // softmax_scale * log2(e)
  const int* page_table;
  const int* seq_lens;
  const int* q_start;
  const int* idx;
  __nv_bfloat16* out;
  float* lse;
  int* status;
  float* ws_o;     // [n_q][2][splits][128][256] normalised partial outputs
  float* ws_lse;   // [n_q][2][splits][128] partial log2-sum-exp
  int* ws_count;   // [n_q][2] arrival counters (zero between calls)
  const __nv_bfloat16* q;
  const __nv_bfloat16* kv;
#ifdef DSA_TEST_HOOKS
  int stall;       // test build: CTA 0's MMA thread waits on a barrier nothing arrives on
#endif
};

// Shared memory.  The TMA-staged value columns of Q[:, D_r] (4 boxes of 128 heads x 128 B, 64 KiB)
// land in the score-exchange and P buffers, which are idle until Q has moved into TMEM; the rope
// columns of Q stay in shared memory (A operand of the two rope k-steps), as does P (A operand of
// P.V).  The total is exactly the 227 KiB a CTA may use (with 1 KiB of alignment slack).
struct Layout {
  static constexpr int stages = 0;
  static constexpr int xbuf = stages + kStages * kTileBytes;   // [2][8 chunks][128 heads] x 16 B
  static constexpr int pbuf = xbuf + 2 * 8 * kHeads * 16;      // P[2]: 128 heads x 128 B, SW128
  static constexpr int qrope = pbuf + 2 * kHeads * 128;  // Q rope half: 128 x 64 B, 64-byte swizzle
  static constexpr int rows = qrope + kHeads * kRopeHalf * 2;
  static constexpr int qstage = xbuf;                    // 64 KiB: xbuf + pbuf
  static constexpr int mxr = rows + kMaxRows * 4;       // [2][128] the peer's row maxima; at the
                                                         // end its partial row sums
  static constexpr int mref = mxr + 2 * kHeads * 4;     // [128] reference maxima between teams
  static constexpr int ctl = mref + kHeads * 4;
  static constexpr int total = ctl + 512;
  // epilogue, in the idle ring: staged O rows [0, 128 KiB), then the lse of every head and the
  // other split's lse of the heads this CTA finalises (cluster merge), then 1/l of every head
  static constexpr int lsebuf = stages + kHeads * 1024;
  static constexpr int invbuf = lsebuf + 192 * 4;
};
static_assert(2 * 8 * kHeads * 16 + 2 * kHeads * 128 >= 4 * kHeads * 128, "Q staging");
static_assert(Layout::invbuf + 128 * 4 <= Layout::stages + kStages * kTileBytes, "lse in the ring");

struct Ctl {
  uint64_t qbar, q_tmem;
  uint64_t full[kStages], empty[kStages];
  uint64_t s_full[2], s_free[2];
  uint64_t xfull[2];   // the peer's partial S of our columns has arrived in xbuf[b]
  uint64_t xfree[2];   // the peer has consumed what we stored into its xbuf[b]
  uint64_t mx[2];      // the peer's row maxima of tile buffer b have arrived in mxr[b]
  uint64_t p_full[2];  // our columns of P buffer b are written (and O rescaled): P.V may run once
  uint64_t p_rem[2];   // ... the peer's columns of P have arrived too
  uint64_t pfree[2];   // the peer's P.V has read its P buffer b: we may store into it again
  uint64_t hand[2];    // team b has left the reference maximum of its latest tile in mref
  uint64_t pv_done[2], drain, fin, mxdone;
#ifdef DSA_TEST_HOOKS
  uint64_t never;      // test build: no thread ever arrives here
#endif
  uint32_t tmem_base;
  int abort;
  int nvalid;          // rows up to the last valid slot; at the end: this CTA merges the splits
  int gather_go;       // the gather poller's verdict of step i in bit i & 1
  int bseq, bcnt, blen;  // the token's sequence: index, ranges that held the token, its length
};
static_assert(sizeof(Ctl) <= 512, "control block");

// Cluster merge (two row splits): workspace slot of (token t, value half r, split s) holding the
// normalised rows of the 64 heads the other split finalises ([64][256] fp32) and their lse.
constexpr int kCmRowFloats = kDvHalf;
DSA_DEV size_t cm_slot(int t, int r, int s) { return ((size_t)t * 2 + r) * 2 + s; }

DSA_DEV int find_seq(const int* q_start, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {  // largest b with q_start[b] <= t
    const int mid = (lo + hi + 1) >> 1;
    if (q_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

DSA_DEV uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x with the hardware approximation (flush-to-zero; 2^-inf = 0).  The weights are rounded to
// bf16 right after, so its ~2-ulp fp32 error is far below what the output keeps.
DSA_DEV float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
DSA_DEV void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed.
DSA_DEV void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Byte offset, within a latent row, of 16-byte chunk ch (< kRowChunks) of half r: 32 value
// chunks, then the 4 chunks of the rope half.
DSA_DEV int row_chunk_offset(int ch, int r) {
  return ch < 32 ? r * (kDvHalf * 2) + ch * 16 : kDv * 2 + r * (kRopeHalf * 2) + (ch - 32) * 16;
}
// Shared-memory offset, within a stage, of chunk ch of tile row rr: value chunks go to box ch/8
// (128-byte swizzle), rope chunks to the rope box (64-byte rows, 64-byte swizzle).
DSA_DEV uint32_t stage_chunk_offset(int ch, int rr) {
  return ch < 32 ? (uint32_t)((ch >> 3) * kBoxBytes + rr * 128 + (((ch & 7) ^ (rr & 7)) << 4))
                 : (uint32_t)(4 * kBoxBytes + rr * 64 + ((((ch - 32) ^ (rr >> 1)) & 3) << 4));
}

// FP8 latent rows: 576 e4m3 codes, one fp32 scale per 128-column tile (5), padding to 608 B.
constexpr int kKv8Row = 608;
// A CTA's part of an FP8 row as staged in the upper part of a ring stage: 256 value codes, 32 rope
// codes and the row's 32 scale bytes (20 chunks of 16 bytes), 64 rows = 20 KiB.
constexpr int kKv8Chunks = 20;
constexpr int kKv8StageRow = 16 * kKv8Chunks;
constexpr int kKv8Stage = kTileBytes - kNT * kKv8StageRow;  // 16 KiB

// Two e4m3 codes (low byte first) times their tile scale: fp32 products rounded to nearest, then
// packed as two bf16 rounded to nearest even.
DSA_DEV uint32_t dequant2(uint32_t codes2, float scale) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)codes2, __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  return pack_bf16(f.x * scale, f.y * scale);
}

// O row of TMEM lane `lane_addr`, columns [col0, col0 + 128), times `alpha`.
DSA_DEV void rescale_o(uint32_t lane_addr, uint32_t col0, float alpha) {
#pragma unroll 1
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t o[32];
    tmem_ld_x32(lane_addr + col0 + (uint32_t)(cc * 32), o);
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
    tmem_st_x16(lane_addr + col0 + (uint32_t)(cc * 32), o);
    tmem_st_x16(lane_addr + col0 + (uint32_t)(cc * 32 + 16), o + 16);
  }
  tmem_st_wait();
}

template <bool KV8>
__global__ void __launch_bounds__(kThreads, 1)
    sfa_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qr,
               const Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from smem_raw by pointer arithmetic so that the compiler
  // keeps the accesses through it in the shared state space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* st_s = smem + Layout::stages;
  uint4* xbuf = reinterpret_cast<uint4*>(smem + Layout::xbuf);
  int* rows_s = reinterpret_cast<int*>(smem + Layout::rows);
  float* mxr = reinterpret_cast<float*>(smem + Layout::mxr);
  float* mref = reinterpret_cast<float*>(smem + Layout::mref);
  float* lsebuf = reinterpret_cast<float*>(smem + Layout::lsebuf);
  float* invbuf = reinterpret_cast<float*>(smem + Layout::invbuf);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + Layout::ctl);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = blockIdx.x & 1;  // == rank in the cluster pair
  const int split = (blockIdx.x >> 1) % p.splits;
  const int t = (blockIdx.x >> 1) / p.splits;
  if (t >= p.n_q) return;  // uniform over the pair
  const uint32_t crank = cluster_rank();
  const uint32_t peer = crank ^ 1u;  // the other value half of this (token, split)
  const int slot0 = split * p.rows_per;
  const int nslot = max(0, min(p.rows_per, p.K - slot0));

  if (tid == 0) {
    mbar_init(&ctl->qbar, 1);
    mbar_init(&ctl->q_tmem, 128);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], kGatherThreads);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {       // buffer b: tiles i with i % 2 == b, score team b
      mbar_init(&ctl->s_full[b], 1);
      mbar_init(&ctl->s_free[b], 128);  // team b
      mbar_init(&ctl->xfull[b], 1);     // one local expect_tx arrival + the peer's stored bytes
      mbar_init(&ctl->xfree[b], 128);   // the peer's team b
      mbar_init(&ctl->mx[b], 1);
      mbar_init(&ctl->p_full[b], 128);  // team b
      mbar_init(&ctl->p_rem[b], 1);
      mbar_init(&ctl->pfree[b], 128);   // the peer's team b
      mbar_init(&ctl->hand[b], 128);    // team b
      mbar_init(&ctl->pv_done[b], 1);
    }
    mbar_init(&ctl->drain, 1);
    mbar_init(&ctl->fin, 1);
    mbar_init(&ctl->mxdone, 256);       // both teams of the peer have read their last maxima
    // The peer's P columns of tiles 0 and 1; the MMA thread, which observes each phase complete,
    // arms the next phase of a buffer when it consumes one.
    mbar_arrive_expect_tx(&ctl->p_rem[0], kPRemBytes);
    mbar_arrive_expect_tx(&ctl->p_rem[1], kPRemBytes);
#ifdef DSA_TEST_HOOKS
    mbar_init(&ctl->never, 1);
#endif
    ctl->abort = 0;
    ctl->nvalid = 0;
    ctl->gather_go = 0;
    ctl->bseq = -1;
    ctl->bcnt = 0;
    ctl->blen = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();  // barriers initialised
  cluster_sync();   // ... in every CTA of the cluster before any remote arrive
  // The launch may overlap the end of the preceding kernel in the stream (programmatic dependent
  // launch): everything above touches only this CTA's resources; no global memory is read
  // before the preceding kernel has completed and its writes are visible.
  griddep_wait();
  if (warp == kMmaWarp && lane == 0 && nslot > 0) {
    // value columns of Q[:, D_r] -> shared memory (moved into TMEM by warps 12-15); issued before
    // the sequence lookup and the row translation below so the load overlaps them
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_qr);
    mbar_arrive_expect_tx(&ctl->qbar, 4 * kHeads * 128 + kHeads * kRopeHalf * 2);
    for (int bx = 0; bx < 4; ++bx)
      tma_load_2d(smem + Layout::qstage + bx * (kHeads * 128), &tm_q, &ctl->qbar,
                  (4 * half + bx) * 64, t * p.H);
    tma_load_2d(smem + Layout::qrope, &tm_qr, &ctl->qbar, kDv + kRopeHalf * half, t * p.H);
  }
  // this split's selected positions: their loads are in flight during the sequence lookup
  constexpr int kPer = kMaxRows / kThreads;
  int j[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int i = u * kThreads + tid;
    j[u] = i < nslot ? p.idx[(size_t)t * p.K + slot0 + i] : -1;
  }
  // the token's sequence in one round of loads: every thread tests one sequence's range of
  // tokens (a binary search over q_start is a chain of dependent loads).  The FP8-cache
  // instantiation runs at the register limit, where the lookup's extra live state cost more
  // (spills in the gather loop) than its saved loads, so it keeps the search.
  int b_seq, len_b;
  if constexpr (!KV8) {
    for (int i = tid; i < p.B; i += kThreads) {
      const int s0 = p.q_start[i], s1 = p.q_start[i + 1], len = p.seq_lens[i];
      if (s0 <= t && t < s1) {
        atomicMax(&ctl->bseq, i);
        atomicAdd(&ctl->bcnt, 1);
        ctl->blen = len;
      }
    }
    __syncthreads();
    b_seq = ctl->bseq;
    len_b = ctl->blen;
  }
  if (KV8 || ctl->bcnt != 1) {  // (or q_start not increasing, or t outside it) the largest b with
                                // q_start[b] <= t
    b_seq = find_seq(p.q_start, p.B, t);
    len_b = p.seq_lens[b_seq];
  }
  const int L = min(len_b, p.max_pages * 64);  // positions the page table covers
  // logical position -> physical row of every slot of this split (-1: empty or invalid): all
  // page-table loads of a thread in flight together
  int last_valid = -1;
  {
    int pg[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u)
      pg[u] = (j[u] >= 0 && j[u] < L) ? p.page_table[(size_t)b_seq * p.max_pages + (j[u] >> 6)] : -1;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = u * kThreads + tid;
      int row = -1;
      if (i < nslot) {
        if (j[u] >= 0) {
          if (j[u] < L && pg[u] >= 0 && pg[u] < p.num_pages)
            row = pg[u] * 64 + (j[u] & 63);
          else if (half == 0)
            report(p.status, kStatusDeviceCheck);
        } else if (j[u] < -1 && half == 0) {
          report(p.status, kStatusDeviceCheck);
        }
        rows_s[i] = row;
        if (row >= 0) last_valid = i;
      }
    }
  }
  // tiles needed: up to the last valid slot (the same in both CTAs of the pair)
  last_valid = __reduce_max_sync(0xffffffffu, last_valid + 1) - 1;
  if (lane == 0 && last_valid >= 0) atomicMax(&ctl->nvalid, last_valid + 1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int ntile = (ctl->nvalid + kNT - 1) / kNT;
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  if (warp < 4 || (warp >= 9 && warp < 12)) {
    // ---------------- gather: 16-byte cp.async of this CTA's 576 bytes of each selected row
    // into the ring, 128-byte swizzled [box][row][128 B] so the tile is a valid tcgen05 operand
    const int g = warp < 4 ? tid : tid - 9 * 32 + 128;  // 0 .. kGatherThreads - 1
    const uint8_t* kv = reinterpret_cast<const uint8_t*>(p.kv);
    // One thread polls each barrier; the other gather warps sleep on a hardware barrier and
    // then read the poller's verdict (bit i & 1 of gather_go, which is not rewritten before
    // every gather thread has passed the next bar.sync, so all of them leave at the same step).
    if constexpr (KV8) {
      // FP8 rows ("Inference Optimization for Kimi K3.1 Pro", section 4: the cache is FP8 with a
      // scale per token and 128-column tile, the attention arithmetic BF16).  The codes and
      // scales this CTA uses (320 of a row's 608 bytes: its 256 value codes, 32 rope codes and
      // the 32 scale bytes) are copied with cp.async into the upper 20 KiB of the tile's stage,
      // and a tile is converted into the swizzled BF16 operand after the next one has been
      // issued, so the copies of two tiles are in flight while the threads convert.
      auto issue = [&](int i, int s) {
        const uint32_t stg = smem_u32(st_s) + (uint32_t)(s * kTileBytes + kKv8Stage);
        for (int c = g; c < kNT * kKv8Chunks; c += kGatherThreads) {
          const int r = c / kKv8Chunks, k = c % kKv8Chunks;
          const int slot = i * kNT + r;
          const int row = slot < nslot ? rows_s[slot] : -1;
          const uint32_t src_off = k < 16 ? (uint32_t)(kDvHalf * half + 16 * k)
                                 : (k < 18 ? (uint32_t)(kDv + kRopeHalf * half + 16 * (k - 16))
                                           : (uint32_t)(kDqk + 16 * (k - 18)));
          const uint8_t* src = row >= 0 ? kv + (size_t)row * kKv8Row + src_off : kv;
          cp_async16(stg + (uint32_t)(r * kKv8StageRow + 16 * k), src, row >= 0 ? 16u : 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      };
      auto convert = [&](int s, bool newer_pending) {
        if (newer_pending)
          asm volatile("cp.async.wait_group 1;" ::: "memory");
        else
          asm volatile("cp.async.wait_group 0;" ::: "memory");
        named_barrier(1, kGatherThreads);  // every thread's copies of tile i have landed
        uint8_t* stage = st_s + (size_t)s * kTileBytes;
        const uint8_t* stg = stage + kKv8Stage;
        uint2 code[kGatherPer];
        float sc[kGatherPer];
#pragma unroll
        for (int k = 0; k < kGatherPer; ++k) {
          const int c = g + k * kGatherThreads;
          code[k] = make_uint2(0u, 0u);
          sc[k] = 0.f;
          if (c < kChunks) {
            const int r = c / kRowChunks, ch = c % kRowChunks;
            const uint8_t* rp = stg + r * kKv8StageRow;
            const int e = ch < 32 ? 8 * ch : kDvHalf + 8 * (ch - 32);  // first of the 8 codes
            const int tile = ch < 32 ? 2 * half + ch / 16 : 4;         // their 128-column tile
            code[k] = *reinterpret_cast<const uint2*>(rp + e);
            sc[k] = *reinterpret_cast<const float*>(rp + 288 + 4 * tile);
          }
        }
        named_barrier(1, kGatherThreads);  // staged bytes are read before the BF16 tile overwrites them
#pragma unroll
        for (int k = 0; k < kGatherPer; ++k) {
          const int c = g + k * kGatherThreads;
          if (c < kChunks) {
            const int r = c / kRowChunks, ch = c % kRowChunks;
            *reinterpret_cast<uint4*>(stage + stage_chunk_offset(ch, r)) =
                make_uint4(dequant2(code[k].x & 0xffffu, sc[k]), dequant2(code[k].x >> 16, sc[k]),
                           dequant2(code[k].y & 0xffffu, sc[k]), dequant2(code[k].y >> 16, sc[k]));
          }
        }
        fence_proxy_async_smem();  // generic-proxy stores -> the tensor core's reads
        mbar_arrive(&ctl->full[s]);
      };
      int issued = 0;
      for (int i = 0; i < ntile; ++i) {
        const int s = i % kStages;
        if (i >= kStages) {
          // a reused stage waits for the P.V that read it
          if (g == 0) {
            const int v = mbar_wait(&ctl->empty[s], ((uint32_t)(i / kStages) & 1u) ^ 1u, abort, p.status) ? 1 : 0;
            volatile int* go = &ctl->gather_go;
            *go = (*go & ~(1 << (i & 1))) | (v << (i & 1));
          }
          named_barrier(1, kGatherThreads);
          if (((*reinterpret_cast<volatile int*>(&ctl->gather_go) >> (i & 1)) & 1) == 0) break;
        }
        issue(i, s);
        issued = i + 1;
        if (i >= 1) convert((i - 1) % kStages, true);
      }
      if (issued == ntile && ntile > 0) convert((ntile - 1) % kStages, false);
    } else {
      for (int i = 0; i < ntile; ++i) {
        const int s = i % kStages;
        if (i >= kStages) {
          // a reused stage waits for the P.V that read it
          if (g == 0) {
            const int v = mbar_wait(&ctl->empty[s], ((uint32_t)(i / kStages) & 1u) ^ 1u, abort, p.status) ? 1 : 0;
            volatile int* go = &ctl->gather_go;
            *go = (*go & ~(1 << (i & 1))) | (v << (i & 1));
          }
          named_barrier(1, kGatherThreads);
          if (((*reinterpret_cast<volatile int*>(&ctl->gather_go) >> (i & 1)) & 1) == 0) break;
        }
        const uint32_t base = smem_u32(st_s) + (uint32_t)(s * kTileBytes);
#pragma unroll
        for (int k = 0; k < kGatherPer; ++k) {
          const int c = g + k * kGatherThreads;
          if (c < kChunks) {
            const int r = c / kRowChunks, ch = c % kRowChunks;
            const int slot = i * kNT + r;
            const int row = slot < nslot ? rows_s[slot] : -1;
            const uint32_t dst = base + stage_chunk_offset(ch, r);
            const uint8_t* src = row >= 0 ? kv + (size_t)row * (kDqk * 2) + row_chunk_offset(ch, half) : kv;
            cp_async16(dst, src, row >= 0 ? 16u : 0u);
          }
        }
        cp_async_arrive_noinc(&ctl->full[s]);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc_qk = idesc_bf16(128, kNT);
      constexpr uint32_t idesc_pv = idesc_bf16(128, kDvHalf, /*b_mn_major=*/true);
      // Descriptors are built once; a k-step only moves the start address (the 14-bit address
      // field cannot carry: every operand lies below 256 KiB).
      const uint64_t st_desc = sdesc_sw128(smem_u32(st_s), 16, 1024);
      const uint64_t v_desc = sdesc_sw128(smem_u32(st_s), kBoxBytes, 1024);
      const uint64_t qr_desc = sdesc_sw64(smem_u32(smem + Layout::qrope), 512);
      const uint64_t rope_desc = sdesc_sw64(smem_u32(st_s) + 4u * kBoxBytes, 512);
      const uint64_t p_desc = sdesc_sw128(smem_u32(smem + Layout::pbuf), 16, 1024);
      bool ok = nslot == 0 || mbar_wait(&ctl->qbar, 0, abort, p.status);  // no TMA left in flight
#ifdef DSA_TEST_HOOKS
      if (p.stall == 2 && blockIdx.x == 0) ok = ok && mbar_wait(&ctl->never, 0, abort, p.status);
#endif
      ok = ok && (ntile == 0 || mbar_wait(&ctl->q_tmem, 0, abort, p.status));
      // Issue whichever is ready: P.V of the oldest tile whose weights are written (needs P; it
      // releases a ring stage) is tested first, then Q.K^T of the next tile (needs its rows and a
      // free S buffer).
      int nqk = 0, npv = 0;
      uint64_t t_idle = 0;
      while (ok && npv < ntile) {
        bool progressed = false;
        if (npv < nqk && mbar_test(&ctl->p_full[npv & 1], (uint32_t)(npv >> 1) & 1u) &&
            mbar_test_cluster(&ctl->p_rem[npv & 1], (uint32_t)(npv >> 1) & 1u)) {
          // our P columns were stored by threads of this CTA, the peer's by st.async: both are
          // read by the tensor core (async proxy)
          fence_proxy_async_smem();
          tc_fence_after();
          const int s = npv % kStages;
          const uint64_t vb = v_desc + (uint64_t)((s * kTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kNT / 16; ++kk) {
            // A = P (K-major, keys [16kk, 16kk+16)); B = V rows [16kk, 16kk+16) x this half's 256
            // value columns, MN-major: 64-column blocks kBoxBytes apart (lbo), 8-row groups 1024
            // bytes apart (sbo)
            mma_f16_ss(tmem + kColO, p_desc + (uint64_t)(((npv & 1) * kHeads * 128 + kk * 32) >> 4),
                       vb + (uint64_t)(kk * 2048 >> 4),
                       idesc_pv, (npv > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&ctl->pv_done[npv & 1]);
          mma_commit(&ctl->empty[s]);
          // the phase of p_rem for tile npv is complete: arm the one of tile npv + 2
          if (npv + 2 < ntile) mbar_arrive_expect_tx(&ctl->p_rem[npv & 1], kPRemBytes);
          ++npv;
          progressed = true;
        }
        if (nqk < ntile && mbar_test(&ctl->full[nqk % kStages], (uint32_t)(nqk / kStages) & 1u) &&
            (nqk < 2 || mbar_test(&ctl->s_free[nqk & 1], (uint32_t)((nqk >> 1) - 1) & 1u))) {
          // the tile was written by cp.async (generic proxy); tcgen05.mma reads it (async proxy)
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sbase = (uint32_t)((nqk % kStages) * kTileBytes);
          const uint32_t d_s = tmem + kColS + (uint32_t)((nqk & 1) * kNT);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {  // the value boxes, A = Q from TMEM
            const uint32_t off = (uint32_t)(kk >> 2) * kBoxBytes + (uint32_t)(kk & 3) * 32u;
            mma_f16_ts(d_s, tmem + kColQ + (uint32_t)kk * 8u, st_desc + ((sbase + off) >> 4), idesc_qk,
                       kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)  // this CTA's rope half, A = Q from shared memory
            mma_f16_ss(d_s, qr_desc + (uint64_t)(kk * 2), rope_desc + (uint64_t)((sbase >> 4) + kk * 2),
                       idesc_qk, 1u);
          mma_commit(&ctl->s_full[nqk & 1]);
          ++nqk;
          progressed = true;
        }
        if (progressed) {
          t_idle = 0;
        } else {
          const uint64_t now = globaltimer();
          if (t_idle == 0) t_idle = now;
          if (*abort) break;
          if (now - t_idle > kWaitLimitNs) {
            *abort = 1;
            report(p.status, kStatusTimeout);
            break;
          }
        }
      }
      mma_commit(&ctl->drain);
      mbar_wait(&ctl->drain, 0, abort, p.status);
    }
    __syncwarp();  // the warp is converged again before the aligned cluster barrier
  } else {
    // ---------------- score warps 4-7 (team 0: even tiles) and 12-15 (team 1: odd tiles), one
    // thread per head row h = TMEM lane (quadrant warp % 4).  The pair splits each 64-row tile by
    // columns: this CTA finalises the softmax of columns [32 half, 32 half + 32) for every head,
    // so the exponentials spread over all four lane quadrants (each served by its own SM
    // sub-partition), and the two teams take alternate tiles, so that one tile's exchanges with
    // the peer overlap the next tile's.  For a tile, a thread:
    //   - sends our partial of the peer's columns of its row to the peer;
    //   - adds the peer's partial of our columns (always S_0 + S_1), masks and scales them;
    //   - exchanges the row maximum of our columns with the peer (both CTAs then hold the same
    //     tile maximum and take the same rescale decisions);
    //   - takes the reference maximum left by the other team's tile, moves it lazily (only
    //     when exceeded by more than 2^8, then rescaling O) and leaves it to the other team;
    //   - writes our columns of P (bf16) into our P buffer and the peer's.
    const int qd = warp & 3;                 // TMEM lane quadrant
    const int team = warp >= 12 ? 1 : 0;     // tiles i with i % 2 == team; also P / xbuf buffer
    const int h = qd * 32 + lane;            // head = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(qd * 32) << 16);
    const uint32_t col_fin = (uint32_t)(kFinCols * half);        // our columns of a tile
    const uint32_t col_snd = (uint32_t)(kFinCols * (half ^ 1));  // the peer's
    const uint32_t peer_xbuf = map_cluster(xbuf, peer);
    const uint32_t peer_pbuf = map_cluster(smem + Layout::pbuf, peer);
    const uint32_t peer_mxr = map_cluster(mxr, peer);
    const uint32_t peer_xfull = map_cluster(&ctl->xfull[team], peer);
    const uint32_t peer_xfree = map_cluster(&ctl->xfree[team], peer);
    const uint32_t peer_mx = map_cluster(&ctl->mx[team], peer);
    const uint32_t peer_prem = map_cluster(&ctl->p_rem[team], peer);
    const uint32_t peer_pfree = map_cluster(&ctl->pfree[team], peer);
    const uint32_t peer_finbar = map_cluster(&ctl->fin, peer);
    const uint32_t peer_mxdone = map_cluster(&ctl->mxdone, peer);
    const int b = team;
    if (team == 1 && ntile > 0) {
      // Q[t][h][value columns of D_r] -> TMEM columns kColQ.. (two bf16 per 32-bit column) from
      // the TMA-staged boxes (128-byte swizzled); heads >= H are 0.
      const bool ok = mbar_wait(&ctl->qbar, 0, abort, p.status);
      (void)ok;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t r[32];
        const uint8_t* box = smem + Layout::qstage + cc * (kHeads * 128) + h * 128;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = h < p.H ? *reinterpret_cast<const uint4*>(box + ((v ^ (h & 7)) << 4))
                                  : make_uint4(0u, 0u, 0u, 0u);
          r[4 * v] = x.x; r[4 * v + 1] = x.y; r[4 * v + 2] = x.z; r[4 * v + 3] = x.w;
        }
        tmem_st_x16(lane_addr + kColQ + (uint32_t)(cc * 32), r);
        tmem_st_x16(lane_addr + kColQ + (uint32_t)(cc * 32 + 16), r + 16);
      }
      if (h >= p.H) {  // padded heads: zero rope row (the staged rows belong to the next token)
#pragma unroll
        for (int v = 0; v < 4; ++v)
          *reinterpret_cast<uint4*>(smem + Layout::qrope + h * (kRopeHalf * 2) + v * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ctl->q_tmem);
    }
    if (ntile > b) {
      // Our exchange and P buffers hold the staged Q until it is in TMEM; then the peer may
      // store into our exchange buffer of this team (its initial credit).
      mbar_wait(&ctl->q_tmem, 0, abort, p.status);
      mbar_arrive_remote_relaxed(peer_xfree);
    }
    // this team's sums over our columns of the bf16 weights P.V uses (normalisation) and of the
    // unrounded weights (log-sum-exp), relative to the reference m_ref
    float m_ref = -INFINITY, l_sum = 0.f, l_exact = 0.f;
    for (int i = team; i < ntile; i += 2) {
      const uint32_t ph = (uint32_t)(i >> 1) & 1u;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&ctl->s_full[b], ph, abort, p.status));
      if (!ok) break;
      uint32_t sr[32], sp[32];
      tc_fence_after();
      tmem_ld_x32(lane_addr + kColS + (uint32_t)(b * kNT) + col_fin, sr);
      tmem_ld_x32(lane_addr + kColS + (uint32_t)(b * kNT) + col_snd, sp);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&ctl->s_free[b]);
      if (h == 0) {  // (this thread observed the previous phases of both complete)
        mbar_arrive_expect_tx(&ctl->xfull[b], kXBytes);
        mbar_arrive_expect_tx(&ctl->mx[b], kMxBytes);
      }
      // our partial of the peer's columns -> the peer's xbuf[b], chunk k of 4 columns at
      // [b][k][head] (a warp stores 512 contiguous bytes per chunk)
      ok = __all_sync(0xffffffffu, mbar_wait<true>(&ctl->xfree[b], ph, abort, p.status));
      if (!ok) break;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        st_async_v4(peer_xbuf + (uint32_t)(((b * 8 + k) * kHeads + h) * 16),
                    make_uint4(sp[4 * k], sp[4 * k + 1], sp[4 * k + 2], sp[4 * k + 3]), peer_xfull);
      // validity of our 32 slots of the tile (one row-table entry per lane)
      const int slot = i * kNT + (int)col_fin + lane;
      const uint32_t vm = __ballot_sync(0xffffffffu, slot < nslot && rows_s[slot] >= 0);
      ok = __all_sync(0xffffffffu, mbar_wait<true>(&ctl->xfull[b], ph, abort, p.status));
      if (!ok) break;
      // z = (S_0 + S_1) * scale * log2(e) for valid slots, -inf for empty ones
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // independent chains
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 o = xbuf[(b * 8 + k) * kHeads + h];
        const uint32_t ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = 4 * k + e;
          const float a = __uint_as_float(sr[col]), b2 = __uint_as_float(ov[e]);
          const float sv = half == 0 ? a + b2 : b2 + a;
          const bool valid = (vm >> col) & 1u;
          const float z = valid ? sv * p.scale_log2 : -INFINITY;
          sr[col] = __float_as_uint(z);
          m4[e] = fmaxf(m4[e], z);
        }
      }
      const float mk = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      mbar_arrive_remote_relaxed(peer_xfree);  // our xbuf[b] may be refilled
      // the tile's row maximum: ours to the peer, the peer's back
      st_async_b32(peer_mxr + (uint32_t)((b * kHeads + h) * 4), __float_as_uint(mk), peer_mx);
      ok = __all_sync(0xffffffffu, mbar_wait<true>(&ctl->mx[b], ph, abort, p.status));
      if (!ok) break;
      const float mt = fmaxf(mk, mxr[b * kHeads + h]);
      // the reference maximum after the previous tile (the other team's)
      float m_cur = -INFINITY;
      if (i >= 1) {
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->hand[b ^ 1], (uint32_t)((i - 1) >> 1) & 1u,
                                               abort, p.status));
        if (!ok) break;
        m_cur = mref[h];
      }
      // lazy rescale: move the reference only when it is exceeded by more than 2^8 (the same
      // decision in both CTAs: both see the same maximum)
      const bool need = mt > m_cur + kRescaleLog2;
      const float m_new = need ? mt : m_cur;
      mref[h] = m_new;
      mbar_arrive(&ctl->hand[b]);  // the other team's next tile may take it
      const bool resc = need && m_cur != -INFINITY;  // O holds weights of an older reference
      if (__any_sync(0xffffffffu, resc)) {  // implies i >= 1
        ok = __all_sync(0xffffffffu, mbar_wait(&ctl->pv_done[b ^ 1], (uint32_t)((i - 1) >> 1) & 1u,
                                               abort, p.status));
        if (!ok) break;
        tc_fence_after();
        const float alpha = resc ? exp2f(m_cur - m_new) : 1.f;
        rescale_o(lane_addr, kColO, alpha);
        rescale_o(lane_addr, kColO + 128u, alpha);
      }
      if (m_ref != m_new) {  // this team's sums follow the reference
        if (m_ref != -INFINITY) {
          const float f = exp2f(m_ref - m_new);
          l_sum *= f;
          l_exact *= f;
        }
        m_ref = m_new;
      }
      uint32_t pk[16];
      float ls[2] = {0.f, 0.f}, le[2] = {0.f, 0.f};  // independent chains
#pragma unroll
      for (int cc = 0; cc < 16; ++cc) {
        const float p0 = m_ref == -INFINITY ? 0.f : fast_exp2(__uint_as_float(sr[2 * cc]) - m_ref);
        const float p1 = m_ref == -INFINITY ? 0.f : fast_exp2(__uint_as_float(sr[2 * cc + 1]) - m_ref);
        pk[cc] = pack_bf16(p0, p1);
        const __nv_bfloat162 r = *reinterpret_cast<const __nv_bfloat162*>(&pk[cc]);
        ls[cc & 1] += __bfloat162float(r.x) + __bfloat162float(r.y);
        le[cc & 1] += p0 + p1;
      }
      l_sum += ls[0] + ls[1];
      l_exact += le[0] + le[1];
      if (i >= 2) {
        // P buffer b was read by the P.V two tiles back: ours (the peer may write its columns
        // into it again), and the peer's (it says so)
        ok = mbar_wait(&ctl->pv_done[b], (uint32_t)((i - 2) >> 1) & 1u, abort, p.status);
        mbar_arrive_remote_relaxed(peer_pfree);
        ok = mbar_wait<true>(&ctl->pfree[b], (uint32_t)((i >> 1) - 1) & 1u, abort, p.status) && ok;
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      // P row h, our columns = 16-byte chunks 4 half .. 4 half + 3 of the 128-byte row (the A
      // operand of P.V, 128-byte swizzle), into our buffer and the peer's
      const uint32_t row_off = (uint32_t)(b * (kHeads * 128) + h * 128);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint32_t off = row_off + (uint32_t)((((4 * half + v) ^ (h & 7))) << 4);
        const uint4 val = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        *reinterpret_cast<uint4*>(smem + Layout::pbuf + off) = val;
        st_async_v4(peer_pbuf + off, val, peer_prem);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ctl->p_full[b]);
    }
    // we have read our last maxima: the peer may now store its row sums over them
    mbar_arrive_remote_relaxed(peer_mxdone);
    // Row sums of each head over all columns: both teams' (at the final reference) and the
    // peer's, added in the same order in both CTAs (team 0 first, CTA 0 first), so both
    // normalise with the same 1/l and report the same lse.
    named_barrier(3, 256);  // both teams are done: the final reference is in mref
    const float m_fin = ntile > 0 ? mref[h] : -INFINITY;
    if (m_ref != m_fin && m_ref != -INFINITY) {
      const float f = exp2f(m_ref - m_fin);
      l_sum *= f;
      l_exact *= f;
    }
    float2* team_sums = reinterpret_cast<float2*>(xbuf);  // idle: every partial was consumed
    if (team == 1) team_sums[h] = make_float2(l_sum, l_exact);
    named_barrier(3, 256);
    float inv = 0.f, lse2 = -INFINITY;
    if (team == 0) {
      const float2 t1 = team_sums[h];
      l_sum = l_sum + t1.x;
      l_exact = l_exact + t1.y;
      if (h == 0) mbar_arrive_expect_tx(&ctl->fin, kFinBytes);
      // the peer has read its last maxima from the buffer our sums go to
      bool ok = ntile == 0 || mbar_wait<true>(&ctl->mxdone, 0, abort, p.status);
      if (ok) {
        st_async_b32(peer_mxr + (uint32_t)(h * 4), __float_as_uint(l_sum), peer_finbar);
        st_async_b32(peer_mxr + (uint32_t)((kHeads + h) * 4), __float_as_uint(l_exact), peer_finbar);
      }
      ok = ok && mbar_wait<true>(&ctl->fin, 0, abort, p.status);
      if (ok) {
        const float ls_p = mxr[h], le_p = mxr[kHeads + h];
        const float Ls = half == 0 ? l_sum + ls_p : ls_p + l_sum;
        const float Le = half == 0 ? l_exact + le_p : le_p + l_exact;
        inv = Ls > 0.f ? 1.f / Ls : 0.f;
        lse2 = Le > 0.f ? m_fin + log2f(Le) : -INFINITY;
      }
    }
    // the last P.V has landed in O (and every gathered tile has been consumed: the ring is idle)
    if (ntile > 0) {
      const bool ok =
          mbar_wait(&ctl->pv_done[(ntile - 1) & 1], (uint32_t)((ntile - 1) >> 1) & 1u, abort, p.status);
      (void)__all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    if (team == 0) {
      invbuf[h] = inv;
      lsebuf[h] = lse2;
    }
    named_barrier(3, 256);
    if (team == 1) {
      inv = invbuf[h];
      lse2 = lsebuf[h];
    }
    const int c = team;  // value columns [128c, 128c + 128) of the head
    // ---------------- epilogue: the normalised O row (this thread: its 128 value columns) goes
    // into the (now idle) ring, 16-byte chunk k of row h at chunk k ^ (h & 31) so that a warp's
    // stores spread over the banks; all threads then copy the tile out with coalesced stores
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t o[32];
      if (ntile > 0) {
        tmem_ld_x32(lane_addr + kColO + (uint32_t)(128 * c + 32 * cc), o);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = 0u;
      }
      if (p.splits == 1) {  // bf16 rows of 512 B: chunks 16c + 4cc .. +3
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
          w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
          w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
          w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
          *reinterpret_cast<uint4*>(st_s + h * 512 + (((16 * c + 4 * cc + v) ^ (h & 31)) << 4)) = w;
        }
      } else if (p.cluster_merge && (h >> 6) != split) {
        // a head the other split finalises: its row goes to our workspace slot for it (L2), while
        // the cluster's CTAs are still finishing (the 20-byte-per-clock distributed shared
        // memory would take longer)
        float* dst = p.ws_o + cm_slot(t, half, split) * kCmRowFloats * 64 + (h & 63) * kDvHalf +
                     128 * c + 32 * cc;
#pragma unroll
        for (int v = 0; v < 8; ++v)
          __stcg(reinterpret_cast<float4*>(dst + 4 * v),
                 make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                             __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv));
      } else {  // fp32 rows of 1 KiB: chunks 32c + 8cc .. +7
#pragma unroll
        for (int v = 0; v < 8; ++v)
          *reinterpret_cast<float4*>(st_s + h * 1024 + (((32 * c + 8 * cc + v) ^ (h & 31)) << 4)) =
              make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                          __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
      }
    }
    if (team == 0) {
      if (p.splits == 1) {
        if (half == 0 && h < p.H && p.lse) p.lse[(size_t)t * p.H + h] = lse2 * 0.69314718055994531f;
      } else if (!p.cluster_merge) {
        const size_t unit = ((size_t)t * 2 + half) * p.splits + split;
        __stcg(p.ws_lse + unit * kHeads + h, lse2);
      } else if ((h >> 6) != split) {
        __stcg(p.ws_lse + cm_slot(t, half, split) * 64 + (h & 63), lse2);
      }
    }
  }
  tc_fence_before();
  cluster_sync();  // also: no remote access to either CTA's shared memory after this point
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
  // coalesced copy of the staged O tile: a warp writes 512 contiguous bytes
  if (p.splits == 1) {
#pragma unroll 4
    for (int idx = tid; idx < kHeads * 32; idx += kThreads) {
      const int row = idx >> 5, c = idx & 31;
      if (row < p.H)
        *reinterpret_cast<uint4*>(p.out + ((size_t)t * p.H + row) * kDv + half * kDvHalf + c * 8) =
            *reinterpret_cast<const uint4*>(st_s + row * 512 + ((c ^ (row & 31)) << 4));
    }
    return;
  }
  if (p.cluster_merge) {
    // Split s of this half finalises heads [64s, 64s + 64): its own rows of them are staged in
    // the ring, the other split's are in that split's workspace slot (written before the cluster
    // barrier, whose release/acquire orders them before these loads); the two normalised
    // partials combine by their lse, split 0's term first.
    const int h0 = 64 * split;
    const size_t oth = cm_slot(t, half, split ^ 1);
    // thread -> (4 value columns, 8 heads): a warp reads 512 contiguous bytes of a row per load;
    // all eight loads of a thread and the lse loads below are in flight together
    const float* src = p.ws_o + oth * kCmRowFloats * 64;
    const int c = tid & 63, hb = tid >> 6;
    float4 ov[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      ov[k] = __ldcg(reinterpret_cast<const float4*>(src + (hb + 8 * k) * kDvHalf + 4 * c));
    float* w0s = reinterpret_cast<float*>(smem + Layout::xbuf);  // idle now: [64] and [64]
    float* w1s = w0s + 64;
    if (tid < 64) {
      const float lo = lsebuf[h0 + tid], lp = __ldcg(p.ws_lse + oth * 64 + tid);
      const float M = fmaxf(lo, lp);
      const float wo = lo == -INFINITY ? 0.f : exp2f(lo - M);
      const float wp = lp == -INFINITY ? 0.f : exp2f(lp - M);
      const float W = wo + wp, inv = W > 0.f ? 1.f / W : 0.f;
      w0s[tid] = (split == 0 ? wo : wp) * inv;
      w1s[tid] = (split == 0 ? wp : wo) * inv;
      if (half == 0 && h0 + tid < p.H && p.lse)
        p.lse[(size_t)t * p.H + h0 + tid] = W > 0.f ? (M + log2f(W)) * 0.69314718055994531f : -INFINITY;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int hr = hb + 8 * k, h = h0 + hr;
      const float4 a = *reinterpret_cast<const float4*>(st_s + h * 1024 + ((c ^ (h & 31)) << 4));
      const float4 x0 = split == 0 ? a : ov[k], x1 = split == 0 ? ov[k] : a;
      const float w0 = w0s[hr], w1 = w1s[hr];
      if (h < p.H) {
        uint2 v;
        v.x = pack_bf16(w0 * x0.x + w1 * x1.x, w0 * x0.y + w1 * x1.y);
        v.y = pack_bf16(w0 * x0.z + w1 * x1.z, w0 * x0.w + w1 * x1.w);
        *reinterpret_cast<uint2*>(p.out + ((size_t)t * p.H + h) * kDv + half * kDvHalf + 4 * c) = v;
      }
    }
    return;
  }
  {
    const size_t unit = ((size_t)t * 2 + half) * p.splits + split;
    float* po = p.ws_o + unit * kHeads * kDvHalf;
#pragma unroll 4
    for (int idx = tid; idx < kHeads * 64; idx += kThreads) {
      const int row = idx >> 6, c = idx & 63;
      __stcg(reinterpret_cast<float4*>(po + row * kDvHalf + c * 4),
             *reinterpret_cast<const float4*>(st_s + row * 1024 + ((c ^ (row & 31)) << 4)));
    }
  }
  __threadfence();  // every thread's partial stores are visible before the arrival count
  __syncthreads();

  // ---------------- last CTA of (token, half) merges the split partials
  if (tid == 0) {
    __threadfence();
    const int prev = atomicAdd(&p.ws_count[t * 2 + half], 1);
    ctl->nvalid = prev == p.splits - 1;
    if (ctl->nvalid) p.ws_count[t * 2 + half] = 0;  // ready for the next call
  }
  __syncthreads();
  if (!ctl->nvalid) return;
  __threadfence();
  const size_t unit0 = ((size_t)t * 2 + half) * p.splits;
  // Coalesced merge: thread -> (4 value columns c4, heads h0 + 8k); a warp reads 512 contiguous
  // bytes of one head row per load.
  float* wgt = reinterpret_cast<float*>(st_s);  // [splits][128] merge weights (ring is free now)
  float* winv = wgt + p.splits * kHeads;        // [128] 1 / sum of weights
  if (tid < kHeads) {
    const int h = tid;
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, __ldcg(p.ws_lse + (unit0 + s) * kHeads + h));
    float W = 0.f;
    for (int s = 0; s < p.splits; ++s) {
      const float ls = __ldcg(p.ws_lse + (unit0 + s) * kHeads + h);
      const float w = (M == -INFINITY || ls == -INFINITY) ? 0.f : exp2f(ls - M);
      wgt[s * kHeads + h] = w;
      W += w;
    }
    winv[h] = W > 0.f ? 1.f / W : 0.f;
    if (half == 0 && h < p.H && p.lse)
      p.lse[(size_t)t * p.H + h] = W > 0.f ? (M + log2f(W)) * 0.69314718055994531f : -INFINITY;
  }
  __syncthreads();
  const int c4 = (tid & 63) * 4, h0 = tid >> 6;
  constexpr int kHeadStep = kThreads / 64;      // 8 head groups
  constexpr int kBatch = 8;                     // heads per thread with loads in flight together
#pragma unroll 1
  for (int hb = h0; hb < kHeads; hb += kHeadStep * kBatch) {
    float4 acc[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
    for (int s = 0; s < p.splits; ++s) {
      float4 x[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        x[k] = __ldcg(reinterpret_cast<const float4*>(
            p.ws_o + ((unit0 + s) * kHeads + hb + k * kHeadStep) * kDvHalf + c4));
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float w = wgt[s * kHeads + hb + k * kHeadStep];
        acc[k].x = fmaf(w, x[k].x, acc[k].x);
        acc[k].y = fmaf(w, x[k].y, acc[k].y);
        acc[k].z = fmaf(w, x[k].z, acc[k].z);
        acc[k].w = fmaf(w, x[k].w, acc[k].w);
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int h = hb + k * kHeadStep;
      if (h < p.H) {
        const float inv = winv[h];
        uint2 v;
        v.x = pack_bf16(acc[k].x * inv, acc[k].y * inv);
        v.y = pack_bf16(acc[k].z * inv, acc[k].w * inv);
        *reinterpret_cast<uint2*>(p.out + ((size_t)t * p.H + h) * kDv + half * kDvHalf + c4) = v;
      }
    }
  }
}

// ---------------------------------------------------------------- host side

struct Plan {
  int splits, rows_per;
  bool cluster_merge;  // two splits of a token in one cluster of 4, merged through the workspace
};

static Plan plan(const dsa_sfa_args& a, bool prefill, int sm_count) {
  Plan pl;
  int splits = 1;
  if (!prefill) {
    const int target = std::max(1, (sm_count + 2 * a.n_q - 1) / (2 * std::max(1, a.n_q)));
    splits = std::max(1, std::min(target, (a.K + kNT - 1) / kNT));
    // never more than the CTAs one wave holds
    while (splits > 1 && 2LL * a.n_q * splits > sm_count) --splits;
  }
  if (!prefill && a.row_splits > 0) splits = std::min(a.row_splits, (a.K + kNT - 1) / kNT);
  int rows_per = ((a.K + splits - 1) / splits + kNT - 1) / kNT * kNT;
  while (rows_per > kMaxRows) {  // K up to 2048 always fits one split
    ++splits;
    rows_per = ((a.K + splits - 1) / splits + kNT - 1) / kNT * kNT;
  }
  splits = (a.K + rows_per - 1) / rows_per;
  pl.splits = splits;
  pl.rows_per = rows_per;
  pl.cluster_merge = splits == 2;
  return pl;
}

// Workspace: [units][rows][256] fp32 partial rows, then [units][rows] lse, then n_q * 2 arrival
// counters (used with three or more splits; zero between calls).  Three or more splits: a unit is
// (token, value half, split) with all 128 rows; two splits (cluster merge): 64 rows, those of the
// heads the other split finalises.
static size_t ws_bytes(const dsa_sfa_args& a, const Plan& pl) {
  if (pl.splits <= 1) return 0;
  const size_t units = (size_t)a.n_q * 2 * pl.splits;
  const size_t rows = pl.cluster_merge ? 64 : kHeads;
  size_t bytes = units * rows * kDvHalf * 4;     // partial o
  bytes += units * rows * 4;                      // partial lse
  bytes = (bytes + 255) / 256 * 256;
  bytes += (size_t)a.n_q * 2 * 4;                 // counters
  return (bytes + 255) / 256 * 256;
}

}  // namespace sfa

size_t sfa_workspace_bytes(const dsa_sfa_args& a) {
  DeviceInfo dev;
  std::string err;
  const int sms = device_info(dev, err) ? dev.sm_count : 152;
  return sfa::ws_bytes(a, sfa::plan(a, false, sms));
}

dsa_status launch_sfa(const dsa_sfa_args& a, bool prefill, cudaStream_t stream, std::string& err) {
  using namespace sfa;
  DeviceInfo dev;
  if (!device_info(dev, err)) return DSA_ERR_CUDA;
  const Plan pl = plan(a, prefill, dev.sm_count);
  const size_t need = ws_bytes(a, pl);
  if (need > 0 && (a.workspace == nullptr || a.workspace_bytes < need)) {
    err = "sfa: workspace of " + std::to_string(need) + " bytes required (got " +
          std::to_string(a.workspace_bytes) + ")";
    return DSA_ERR_INVALID_ARG;
  }
  Params p;
  p.B = a.B;
  p.n_q = a.n_q;
  p.H = a.H;
  p.K = a.K;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.splits = pl.splits;
  p.rows_per = pl.rows_per;
  p.cluster_merge = pl.cluster_merge ? 1 : 0;
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.q_start = a.q_start;
  p.idx = a.idx;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.status = a.status;
  p.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  p.kv = reinterpret_cast<const __nv_bfloat16*>(a.kv_pool);
#ifdef DSA_TEST_HOOKS
  p.stall = g_test_stall;
#endif
  if (need > 0) {
    const size_t units = (size_t)a.n_q * 2 * pl.splits;
    const size_t rows = pl.cluster_merge ? 64 : kHeads;
    uint8_t* ws = reinterpret_cast<uint8_t*>(a.workspace);
    p.ws_o = reinterpret_cast<float*>(ws);
    p.ws_lse = reinterpret_cast<float*>(ws + units * rows * kDvHalf * 4);
    const size_t cnt_off = ((units * rows * kDvHalf * 4 + units * rows * 4) + 255) / 256 * 256;
    p.ws_count = reinterpret_cast<int*>(ws + cnt_off);
  } else {
    p.ws_o = nullptr;
    p.ws_lse = nullptr;
    p.ws_count = nullptr;
  }
  if (a.n_q == 0) return DSA_OK;

  const bool kv8 = a.kv_dtype == DSA_FP8_E4M3;

  CUtensorMap tm_q, tm_qr;
  if (!encode_tmap_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kDqk, (uint64_t)a.n_q * a.H,
                      kDqk * 2, 64, kHeads, CU_TENSOR_MAP_SWIZZLE_128B, err))
    return DSA_ERR_CUDA;
  if (!encode_tmap_2d(&tm_qr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kDqk, (uint64_t)a.n_q * a.H,
                      kDqk * 2, kRopeHalf, kHeads, CU_TENSOR_MAP_SWIZZLE_64B, err))
    return DSA_ERR_CUDA;
  const int smem = Layout::total + 1024;
  auto kern = kv8 ? sfa_kernel<true> : sfa_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "sfa: set shared memory size", err);
  const unsigned grid = (unsigned)(a.n_q * 2 * pl.splits);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  // the two value halves of a (token, split); with a cluster merge both splits of a token
  attr[0].val.clusterDim.x = pl.cluster_merge ? 4 : 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the CTAs may start (barriers, TMEM, cluster handshake) while the preceding kernel finishes
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, tm_q, tm_qr, p);
  if (e != cudaSuccess) return cuda_fail(e, "sfa: launch", err);
  return DSA_OK;
}

}  // namespace dsa
