// li_topk.cu -- fused Lightning Indexer: score contraction on tcgen05 tensor cores, head-weighted
// ReLU reduction in the epilogue, and an exact cluster-wide radix top-K select in shared memory.
// Only the selected positions leave the chip.
//
// Method: "Inference Optimization for Kimi K3.1 Pro: Decoding Architecture Evolution and Systems
// Engineering Practices", section 1 (DSA steps 1-2: indexer scoring with head weights, top-K) and
// section 2 (Operator-Level Deep Fusion: score, head weighting and top-K in one kernel, scores
// kept on chip, indices then drive paged reads); "Day0 Inference Adaptation for Next-Gen LLMs ...
// CANN", section 3.1 (the indexer reads the paged key cache directly; prefill and decode, BF16
// and quantised paths).
//
// Work decomposition.  One thread-block cluster of C CTAs serves one (sequence, group of T query
// tokens).  CTA r of the cluster owns the key positions [r*chunk, (r+1)*chunk) of the sequence:
//   streaming phase  warp 0 issues TMA loads of two 64-row key pages per 128-key tile (page ids
//                    resolved through the page table), warp 1 issues tcgen05.mma
//                    D[128 keys x T*H_I] = K_tile . Q^T into a double-buffered TMEM accumulator,
//                    warps 4..7 and 8..11 (one per accumulator buffer; one TMEM lane = one key per
//                    thread) apply ReLU, the head weights and the head sum, mask by causality and
//                    length, store an order-preserving 32-bit key of each score in shared memory
//                    and build the histogram of its top 11 bits;
//   select phase     every CTA reads the cluster's histograms over distributed shared memory and
//                    finds the bin of the K-th key.  Usually the cluster's keys in that bin are few
//                    enough to gather: each CTA lists its own, one cluster barrier publishes the
//                    lists, and every CTA resolves the remaining 21 bits locally.  Otherwise two
//                    more cluster-wide radix passes (11 and 10 bits) follow.  Every CTA derives
//                    the same K-th key and the number of ties to take; per-warp counts give each
//                    warp its output offset and tie quota (ties go to the lowest positions; CTAs
//                    and warps own ascending position ranges), and a packed warp-scan compaction
//                    writes the positions in ascending order.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace li {

constexpr int kThreads = 384;       // 12 warps: 0 TMA, 1 MMA, 4-7 and 8-11 two epilogue groups
constexpr int kHistThreads = 256;   // threads that own 8 histogram bins each in the select
constexpr int kTileKeys = 128;
constexpr int kHistWords = 1024;  // 2048 radix bins, two 16-bit counters per 32-bit word
constexpr int kMaxCluster = 16;
constexpr int kCtlBytes = 2560;   // shared control block (mbarriers, counters), sizeof(Ctl) rounded up
// Sequences longer than kUnitSpan positions (decode and two-token groups) are split into units
// of at most one cluster's span; the unit merge sorts units x K candidates in shared memory.
constexpr int kUnitSpan = 32768;
constexpr int kMaxUnitCand = 16384;
constexpr int kMaxUnitSeqs = 256;

struct Params {
  int B, n_q, K, max_pages, num_pages;
  int groups;  // token groups per sequence
  int chunk;   // key positions per CTA at most (multiple of 128; sizes the shared memory)
  int C;       // cluster size
  int units;   // position units per sequence at most (1: one cluster covers a whole sequence)
  int nstage;  // TMA ring depth
  const float* w;
  const float* q_scale;
  const float* k_scale;
  const int* page_table;
  const int* seq_lens;
  const int* q_start;
  int* out_idx;
  int* out_cnt;
  int* status;
  const uint8_t* q_sf;  // MXFP8: E8M0 scales of 32-element groups, [n_q][H_I][D_I/32]
  const uint8_t* k_sf;  //        and [num_pages][64][D_I/32]
  float* out_score;     // optional [n_q][K]: the score of every emitted position (-inf padding)
  // units > 1: a sequence of more than C * chunk positions is split into equal units of at most
  // C * chunk positions, one cluster each; such a unit writes its own top-K (ascending
  // positions, -1 padding) and their scores to slot ((b * groups + g) * units + u) * T + tt of
  // these [slots][K] arrays, and the unit merge selects the token's top-K from them
  int* cand_idx;
  float* cand_score;
  const int* items;     // units > 1: [0] = number of items, [1 + k] = (sequence << 8 | unit) of
                        // the k-th cluster, written by the unit plan kernel
#ifdef DSA_TEST_HOOKS
  int stall;            // test build: CTA 0's MMA thread waits on a barrier nothing arrives on
#endif
};

template <int D_I, bool FP8, int H_I, int T, bool MX = false>
struct Cfg {
  static constexpr int kElt = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D_I * kElt;      // 128 or 256
  // key rows arrive as column boxes of kBoxW bytes: 64-byte boxes (64-byte swizzle) for e4m3
  // keys streamed faster than one 128-byte box per row (47.2 against 48.7 µs at decode_32k_fp8;
  // 32-byte boxes took 55 µs)
  static constexpr int kBoxW = FP8 ? 64 : 128;
  static constexpr int kBoxes = kRowBytes / kBoxW;  // key column boxes per row
  static constexpr int kQBoxes = kRowBytes / 128;   // query column boxes (128 bytes) per row
  static constexpr int kKSteps = kRowBytes / 32;    // one MMA consumes 32 bytes of K
  static constexpr int kNCol = (T * H_I < 16) ? 16 : T * H_I;  // MMA N (>= 16 for M = 128)
  static constexpr int kTileBytes = kTileKeys * kRowBytes;
  static constexpr int kQBytes = kNCol * kRowBytes;
  // MXFP8: the E8M0 scale cells follow the two accumulators.  Key side (MMA operand A) of
  // accumulator a: columns kSfA + 4a .. +3, key r of the tile at lane r, column kSfA + 4a + r/32
  // (each lane quadrant reads its own column); query side (operand B): columns kSfB + n/32, MMA
  // column n at lane n%32 of every lane quadrant.  Byte g of a cell is the scale of group g.
  static constexpr int kSfA = 2 * kNCol;
  static constexpr int kSfB = kSfA + 8;
  static constexpr int kTmemNeed = 2 * kNCol + (MX ? 8 + (kNCol + 31) / 32 : 0);
  static constexpr int kTmemCols = (kTmemNeed <= 32)    ? 32
                                   : (kTmemNeed <= 64)  ? 64
                                   : (kTmemNeed <= 128) ? 128
                                   : (kTmemNeed <= 256) ? 256
                                                        : 512;
  static_assert(kNCol % 16 == 0 && kNCol <= 256, "MMA N");
  static_assert(kTmemNeed <= 512, "tensor memory columns");
  static_assert(!MX || (FP8 && D_I == 128), "MXFP8: e4m3 elements, four 32-element groups per row");
  static_assert(T * H_I <= 256, "tokens x heads per group");
};

// Shared memory carve-up (offsets from a 1024-byte aligned base).
struct Layout {
  int stages, q, wts, scores, hist, pages, ctl, total;
  __host__ __device__ Layout(int nstage, int tile_bytes, int q_bytes, int T, int H_I, int chunk) {
    stages = 0;
    q = stages + nstage * tile_bytes;
    wts = q + q_bytes;
    scores = wts + ((T * H_I * 4 + 127) / 128) * 128;
    hist = scores + T * chunk * 4;
    pages = hist + 2 * T * kHistWords * 4;
    ctl = pages + ((2 * (chunk / kTileKeys) * 4 + 127) / 128) * 128;
    total = ctl + kCtlBytes;
  }
};

struct Ctl {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t qbar;
  uint64_t drain;
  uint64_t sinit;  // MXFP8: the first scale cells are in tensor memory
  uint64_t cand_bar;  // candidate path: the other ranks' candidate keys and sure counts are here
#ifdef DSA_TEST_HOOKS
  uint64_t never;  // test build: no thread ever arrives here
#endif
  uint32_t tmem_base;
  int abort;
  uint32_t scan[kThreads / 32];
  uint32_t scan_t[4][kThreads / 32];  // per-token block scans
  int need[4];        // remaining count to select among the current prefix
  uint32_t prefix[4]; // key prefix fixed so far
  int radix[4];       // token needs a radix select (visible > K)
  int need_total[4];  // min(K, visible)
  int cnt_gt[4], cnt_eq[4];  // this CTA's counts (read by the cluster)
  int offset[4], quota[4];
  int found_bin[4], found_need[4];
  int wgt[4][kThreads / 32], weq[4][kThreads / 32];  // per-warp counts above / at the threshold
  int wcnd[4][kThreads / 32];  // candidate path: per-warp candidates in the threshold bin
  // candidate path of the select (see the select phase)
  int cand_total[4];          // keys of the whole cluster in the threshold bin of the first pass
  int few_cnt;                // candidates sharing the 22-bit prefix (local resolution)
  int own_cnt[4];             // this CTA's candidates (read by the cluster)
  int rn[4][kMaxCluster], roff[4][kMaxCluster];    // candidates per rank and their offsets
  int rsure[4][kMaxCluster];  // per rank: keys certainly selected (above the first-pass bin)
  int rgt[4][kMaxCluster], req[4][kMaxCluster];    // per rank: candidates above / at the threshold
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");

// ---- block-level scans over 256 threads ----

// Exclusive suffix sum: sum of v over threads with a larger index.
DSA_DEV uint32_t block_excl_suffix(uint32_t v, uint32_t* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) scratch[warp] = x;
  __syncthreads();
  uint32_t above = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w)
    if (w > warp) above += scratch[w];
  __syncthreads();
  return above + x - v;
}

// The same for NT values per thread at once (one pair of block barriers for all of them).
template <int NT>
DSA_DEV void block_excl_suffix_multi(const uint32_t (&v)[NT], uint32_t (*scratch)[kThreads / 32],
                                     uint32_t (&above)[NT]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) x[n] = v[n];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const uint32_t y = __shfl_down_sync(0xffffffffu, x[n], o);
      if (lane + o < 32) x[n] += y;
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int n = 0; n < NT; ++n) scratch[n][warp] = x[n];
  }
  __syncthreads();
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    uint32_t a = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w)
      if (w > warp) a += scratch[n][w];
    above[n] = a + x[n] - v[n];
  }
  __syncthreads();
}

// Adds the 8 packed 16-bit bins of histogram words h[0..3] of every CTA of the cluster (C CTAs)
// into cnt; the DSMEM loads of up to four CTAs are in flight together.
DSA_DEV void cluster_hist_sum(const uint32_t* h, int C, uint32_t* cnt) {
#pragma unroll 1
  for (int r0 = 0; r0 < C; r0 += 4) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      v[u] = r0 + u < C ? ld_cluster_v4(map_cluster(h, (uint32_t)(r0 + u))) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      cnt[0] += v[u].x & 0xffffu; cnt[1] += v[u].x >> 16;
      cnt[2] += v[u].y & 0xffffu; cnt[3] += v[u].y >> 16;
      cnt[4] += v[u].z & 0xffffu; cnt[5] += v[u].z >> 16;
      cnt[6] += v[u].w & 0xffffu; cnt[7] += v[u].w >> 16;
    }
  }
}

// Inclusive sum over the lanes of the warp.
DSA_DEV uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Set bits of each 4-bit group g < 4 of x, counted into byte g.  Sums of such words over a warp
// stay below 256 per byte, so one scan of the packed word gives four prefix counts at once.
DSA_DEV uint32_t nibble_counts(uint32_t x) {
  uint32_t y = (x & 0xfu) | ((x & 0xf0u) << 4) | ((x & 0xf00u) << 8) | ((x & 0xf000u) << 12);
  y = (y & 0x05050505u) + ((y >> 1) & 0x05050505u);
  return (y & 0x03030303u) + ((y >> 2) & 0x03030303u);
}

// In a 2048-bin histogram (packed 16-bit counters, 1024 words) of this CTA, finds the bin that
// holds the need-th largest key counting from the top bin: ctl->found_bin / found_need.
template <typename CtlT>
DSA_DEV void find_bin_local(const uint32_t* h, uint32_t need, int tt, CtlT* ctl) {
  const int tid = threadIdx.x;
  uint32_t cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (tid < 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(h + 4 * tid);
    cnt[0] = v.x & 0xffffu; cnt[1] = v.x >> 16;
    cnt[2] = v.y & 0xffffu; cnt[3] = v.y >> 16;
    cnt[4] = v.z & 0xffffu; cnt[5] = v.z >> 16;
    cnt[6] = v.w & 0xffffu; cnt[7] = v.w >> 16;
  }
  uint32_t sum = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) sum += cnt[k];
  if (tid == 0) {
    ctl->found_bin[tt] = 0;
    ctl->found_need[tt] = 1;
  }
  const uint32_t above = block_excl_suffix(sum, ctl->scan);
  uint32_t run = above;
#pragma unroll
  for (int k = 7; k >= 0; --k) {
    if (run < need && run + cnt[k] >= need) {
      ctl->found_bin[tt] = 8 * tid + k;
      ctl->found_need[tt] = (int)(need - run);
    }
    run += cnt[k];
  }
  __syncthreads();
}

// ---- the fused kernel ----

template <int D_I, bool FP8, int H_I, int T, bool MX>
__global__ void __launch_bounds__(kThreads, 1)
    li_topk_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                   const Params p) {
  using CF = Cfg<D_I, FP8, H_I, T, MX>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from smem_raw by pointer arithmetic so that the compiler
  // keeps the accesses through it in the shared state space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const Layout lay(p.nstage, CF::kTileBytes, CF::kQBytes, T, H_I, p.chunk);
  uint8_t* stage_base = smem + lay.stages;
  uint8_t* q_s = smem + lay.q;
  float* wts = reinterpret_cast<float*>(smem + lay.wts);
  uint32_t* scores = reinterpret_cast<uint32_t*>(smem + lay.scores);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + lay.hist);
  int* pages = reinterpret_cast<int*>(smem + lay.pages);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + lay.ctl);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)cluster_rank();
  const int cl = blockIdx.x / p.C;
  int b, g, unit;  // sequence, token group, position unit of this cluster
  if (p.units == 1) {
    b = cl / p.groups;
    g = cl % p.groups;
    unit = 0;
  } else {
    // The unit plan kernel ordered the (sequence, unit) items longest first; clusters past the
    // last item exit at once.  (This launch is its programmatic dependent.)
    griddep_wait();
    if (cl >= p.items[0]) return;  // uniform over the cluster
    const int e = p.items[1 + cl];
    b = e >> 8;
    unit = e & 255;
    g = 0;  // units imply one token group per sequence
  }
  if (b >= p.B) return;
  const int qs = p.q_start[b];
  const int n_b = p.q_start[b + 1] - qs;
  const int L = p.seq_lens[b];
  // Cluster-uniform validity (every CTA of the cluster reads the same values).
  if (unit == 0 && g == p.groups - 1 && rank == 0 && tid == 0 && n_b > p.groups * T)
    report(p.status, kStatusDeviceCheck);
  if (n_b < 0 || L < n_b || L > p.units * p.C * p.chunk || L > p.max_pages * 64 || qs < 0 ||
      qs + n_b > p.n_q) {
    if (unit == 0 && rank == 0 && tid == 0) report(p.status, kStatusDeviceCheck);
    return;
  }
  const int nt = min(T, n_b - g * T);
  if (nt <= 0) return;
  // The sequence's units (one unless it is longer than C * chunk) are equal, and within a unit
  // each CTA owns an equal multiple of 128 positions, so short sequences spread over every CTA
  // of their cluster instead of filling the first ones.
  const int n_u = p.units == 1 ? 1 : max(1, (L + p.C * p.chunk - 1) / (p.C * p.chunk));
  if (unit >= n_u) return;
  const int span_u = (L + n_u - 1) / n_u;
  const int chunk = max(kTileKeys, ((span_u + p.C - 1) / p.C + kTileKeys - 1) / kTileKeys * kTileKeys);
  const int u_lo = unit * p.C * chunk;              // the unit's positions: [u_lo, u_hi)
  const int u_hi = min(L, u_lo + p.C * chunk);
  const bool direct = n_u == 1;                     // writes the token's final top-K
  const int t0 = qs + g * T;
  const int pos0 = L - n_b + g * T;  // position of token t0
  const int lo = u_lo + rank * chunk;
  const int lim = min(lo + chunk, u_hi);            // this CTA's positions: [lo, lim)
  const int hi = min(lim, pos0 + nt);
  const int ntile = hi > lo ? (hi - lo + kTileKeys - 1) / kTileKeys : 0;
  const int nscan = min(ntile * kTileKeys, chunk);
  const int npages_seq = (L + 63) / 64;

  // ---------------- setup
  if (tid == 0) {
    for (int s = 0; s < p.nstage; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->tfull[a], 1);
      mbar_init(&ctl->tempty[a], 128);
    }
    mbar_init(&ctl->qbar, 1);
    mbar_init(&ctl->drain, 1);
    mbar_init(&ctl->sinit, 256);  // both epilogue groups
    mbar_init(&ctl->cand_bar, 1);
#ifdef DSA_TEST_HOOKS
    mbar_init(&ctl->never, 1);
#endif
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, CF::kTmemCols);
    tmem_relinquish();
  }
  // physical page of every 64-row half tile of this CTA's range (-1 = past the sequence)
  for (int i = tid; i < 2 * ntile; i += kThreads) {
    const int P = lo / 64 + i;
    int id = -1;
    if (P < npages_seq) {
      id = p.page_table[(size_t)b * p.max_pages + P];
      if (id < 0 || id >= p.num_pages) {
        report(p.status, kStatusDeviceCheck);
        id = 0;  // stay in bounds; results for this token are then unspecified
      }
    }
    pages[i] = id;
  }
  for (int i = tid; i < T * kHistWords; i += kThreads) hist[i] = 0u;  // pass-0 histogram
  for (int i = tid; i < T * H_I; i += kThreads) {
    const int tt = i / H_I, h = i % H_I;
    float v = 0.f;
    if (tt < nt) {
      v = p.w[(size_t)(t0 + tt) * H_I + h];
      if (FP8 && !MX) v *= p.q_scale[(size_t)(t0 + tt) * H_I + h];  // per-token FP8 scale
    }
    wts[i] = v;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  volatile int* abort = &ctl->abort;

  // ---------------- streaming phase: scores of [lo, lo + nscan) into shared memory
  {
    const uint32_t tmem = ctl->tmem_base;
    if (warp == 0 && lane == 0 && ntile > 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_q);
      mbar_arrive_expect_tx(&ctl->qbar, CF::kQBytes);
      for (int bx = 0; bx < CF::kQBoxes; ++bx)
        tma_load_2d(q_s + bx * CF::kNCol * 128, &tm_q, &ctl->qbar, bx * (128 / CF::kElt),
                    t0 * H_I);
      // With one token group per sequence every key row is read by exactly one CTA: stream it
      // with the evict-first L2 policy.  Otherwise other groups re-read it from L2.
      const bool read_once = p.groups == 1;
      const uint64_t pol = l2_policy_evict_first();
      int issued = 0;
      for (int i = 0; i < ntile; ++i) {
        const int s = i % p.nstage;
        const uint32_t ph = (uint32_t)(i / p.nstage) & 1u;
        if (i >= p.nstage && !mbar_wait(&ctl->empty[s], ph ^ 1u, abort, p.status)) break;
        issued = i + 1;
        const int pg0 = pages[2 * i], pg1 = pages[2 * i + 1];
        const uint32_t bytes = (uint32_t)((pg0 >= 0) + (pg1 >= 0)) * CF::kBoxes * 64 * CF::kBoxW;
        mbar_arrive_expect_tx(&ctl->full[s], bytes);
        uint8_t* st = stage_base + (size_t)s * CF::kTileBytes;
        for (int bx = 0; bx < CF::kBoxes; ++bx) {
          // box bx of the tile: [128 keys][kBoxW bytes], the two pages' 64 keys each
          const int x = bx * (CF::kBoxW / CF::kElt);
          uint8_t* sb = st + bx * (128 * CF::kBoxW);
          if (read_once) {
            if (pg0 >= 0) tma_load_2d_hint(sb, &tm_k, &ctl->full[s], x, pg0 * 64, pol);
            if (pg1 >= 0)
              tma_load_2d_hint(sb + 64 * CF::kBoxW, &tm_k, &ctl->full[s], x, pg1 * 64, pol);
          } else {
            if (pg0 >= 0) tma_load_2d(sb, &tm_k, &ctl->full[s], x, pg0 * 64);
            if (pg1 >= 0) tma_load_2d(sb + 64 * CF::kBoxW, &tm_k, &ctl->full[s], x, pg1 * 64);
          }
        }
      }
      // never leave with copies in flight: wait for the last fill of every stage issued (also
      // after an abort: the ring is reused by the select phase)
      for (int i = max(0, issued - p.nstage); i < issued; ++i) {
        const int s = i % p.nstage;
        mbar_wait_drain(&ctl->full[s], (uint32_t)(i / p.nstage) & 1u, p.status);
      }
    } else if (warp == 1 && lane == 0 && ntile > 0) {
      constexpr uint32_t idesc =
          FP8 ? idesc_e4m3(128, CF::kNCol) : idesc_bf16(128, CF::kNCol);
      const uint32_t q_addr = smem_u32(q_s);
      const uint32_t st_addr = smem_u32(stage_base);
      bool ok = mbar_wait(&ctl->qbar, 0, abort, p.status);
#ifdef DSA_TEST_HOOKS
      if (p.stall == 1 && blockIdx.x == 0) ok = ok && mbar_wait(&ctl->never, 0, abort, p.status);
#endif
      if constexpr (MX) ok = ok && mbar_wait(&ctl->sinit, 0, abort, p.status);
      for (int i = 0; ok && i < ntile; ++i) {
        const int s = i % p.nstage;
        const uint32_t ph = (uint32_t)(i / p.nstage) & 1u;
        const int a = i & 1;
        if (!mbar_wait(&ctl->full[s], ph, abort, p.status)) break;
        if (i >= 2 && !mbar_wait(&ctl->tempty[a], ((uint32_t)(i >> 1) & 1u) ^ 1u, abort, p.status))
          break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(a * CF::kNCol);
#pragma unroll
        for (int kk = 0; kk < CF::kKSteps; ++kk) {
          // key side: 32 bytes of K in box kk*32 / kBoxW; query side: in 128-byte box kk*32 / 128
          const uint32_t box = (uint32_t)(kk * 32) / 128u, off = (uint32_t)(kk * 32) % 128u;
          const uint32_t kbox = (uint32_t)(kk * 32) / CF::kBoxW, koff = (uint32_t)(kk * 32) % CF::kBoxW;
          const uint32_t ka = st_addr + (uint32_t)s * CF::kTileBytes + kbox * (128u * CF::kBoxW) + koff;
          const uint64_t ad = CF::kBoxW == 64 ? sdesc_sw64(ka, 512) : sdesc_sw128(ka, 16, 1024);
          const uint64_t bd = sdesc_sw128(q_addr + box * (uint32_t)(CF::kNCol * 128) + off, 16, 1024);
          if constexpr (MX)  // K step kk = scale group kk (byte kk of every scale cell)
            mma_mx_ss(d, ad, bd, idesc_mx_e4m3(128, CF::kNCol, kk, kk),
                      tmem + (uint32_t)(CF::kSfA + 4 * a), tmem + (uint32_t)CF::kSfB, kk > 0 ? 1u : 0u);
          else if (FP8)
            mma_f8_ss(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
          else
            mma_f16_ss(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&ctl->empty[s]);
        mma_commit(&ctl->tfull[a]);
      }
      // all MMAs retired before the accumulator is released
      mma_commit(&ctl->drain);
      mbar_wait(&ctl->drain, 0, abort, p.status);
    } else if (warp >= 4) {
      // Two epilogue groups: warps 4-7 take accumulator 0 (even tiles), warps 8-11 accumulator 1
      // (odd tiles), so two tiles are reduced at once.
      const int grp = (warp - 4) >> 2;
      const int qd = warp & 3;  // TMEM lane quadrant of this warp
      const int row = qd * 32 + lane;
      const uint32_t lanes = tmem + ((uint32_t)(qd * 32) << 16);
      constexpr uint32_t kSfOne = 0x7F7F7F7Fu;  // four E8M0 scales of 1
      // MXFP8: the four group scales of key `row` of tile i (one 32-bit word per key row)
      auto key_sf = [&](int i) -> uint32_t {
        const int pg = pages[2 * i + (row >> 6)];
        return pg >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(p.k_sf) + (size_t)pg * 64 + (row & 63))
                       : kSfOne;
      };
      if constexpr (MX) {
        // Scale cells of this group's first tile and (group 0) of the query heads, before the
        // first MMA; later tiles' key scales are written while the previous tile of the same
        // accumulator is reduced (below).
        tmem_st_x1(lanes + (uint32_t)(CF::kSfA + 4 * grp + qd), grp < ntile ? key_sf(grp) : kSfOne);
        if (grp == 0) {
          for (int c = 0; c * 32 < CF::kNCol; ++c) {
            const int n = c * 32 + lane, tt = n / H_I, h = n % H_I;
            uint32_t v = kSfOne;
            if (n < T * H_I && t0 + tt < p.n_q)
              v = __ldg(reinterpret_cast<const uint32_t*>(p.q_sf) + (size_t)(t0 + tt) * H_I + h);
            tmem_st_x1(lanes + (uint32_t)(CF::kSfB + c), v);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ctl->sinit);
      }
      for (int i = grp; i < ntile; i += 2) {
        const int a = grp;
        const int j = lo + i * kTileKeys + row;
        float ks = 1.f;
        if (FP8 && !MX) {
          const int pg = pages[2 * i + (row >> 6)];
          ks = pg >= 0 ? p.k_scale[(size_t)pg * 64 + (row & 63)] : 0.f;
        }
        const uint32_t sf_next = (MX && i + 2 < ntile) ? key_sf(i + 2) : kSfOne;
        const bool ok = mbar_wait(&ctl->tfull[a], (uint32_t)(i >> 1) & 1u, abort, p.status);
        if (!__all_sync(0xffffffffu, ok)) break;  // tcgen05.ld below needs the whole warp
        tc_fence_after();
        // MMA i has completed, so its scale cells are free: fill them for tile i + 2
        if constexpr (MX) tmem_st_x1(lanes + (uint32_t)(CF::kSfA + 4 * a + qd), sf_next);
        const uint32_t taddr = lanes + (uint32_t)(a * CF::kNCol);
#pragma unroll 1
        for (int tt = 0; tt < T; ++tt) {
          float s;
          if constexpr (H_I == 64) {
            uint32_t r[64];
            tmem_ld_x32(taddr + (uint32_t)(tt * H_I), r);
            tmem_ld_x32(taddr + (uint32_t)(tt * H_I + 32), r + 32);
            tmem_ld_wait();
            // four independent partial sums (the weights are read as float4 broadcasts)
            const float4* w4 = reinterpret_cast<const float4*>(wts + tt * H_I);
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float4 w = w4[q];
              a0 = fmaf(w.x, fmaxf(__uint_as_float(r[4 * q + 0]), 0.f), a0);
              a1 = fmaf(w.y, fmaxf(__uint_as_float(r[4 * q + 1]), 0.f), a1);
              a2 = fmaf(w.z, fmaxf(__uint_as_float(r[4 * q + 2]), 0.f), a2);
              a3 = fmaf(w.w, fmaxf(__uint_as_float(r[4 * q + 3]), 0.f), a3);
            }
            s = (a0 + a1) + (a2 + a3);
          } else {
            uint32_t r[8];
            tmem_ld_x8(taddr + (uint32_t)(tt * H_I), r);
            tmem_ld_wait();
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int h = 0; h < 8; h += 2) {
              a0 = fmaf(wts[tt * H_I + h], fmaxf(__uint_as_float(r[h]), 0.f), a0);
              a1 = fmaf(wts[tt * H_I + h + 1], fmaxf(__uint_as_float(r[h + 1]), 0.f), a1);
            }
            s = a0 + a1;
          }
          if (FP8 && !MX) s *= ks;
          const bool valid = tt < nt && j < lim && j <= pos0 + tt;
          const uint32_t u = valid ? score_key(s) : 0u;
          scores[tt * p.chunk + (j - lo)] = u;
          if (valid) atomicAdd(&hist[tt * kHistWords + (u >> 22)], 1u << (((u >> 21) & 1u) * 16u));
        }
        if constexpr (MX) tmem_st_wait();  // the scale cells of tile i + 2 are written
        tc_fence_before();
        mbar_arrive(&ctl->tempty[a]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(ctl->tmem_base, CF::kTmemCols);
  }
  if (*abort) {
    // A wait of this CTA gave up (DSA_ERR_TIMEOUT is in *status): keys of tiles it did not
    // reduce were never written.  The select still runs -- every CTA of the cluster takes the
    // same cluster barriers -- over no keys of this CTA, so that every shared-memory index it
    // derives stays in bounds; the token's output is unspecified.
    for (int i = tid; i < T * p.chunk; i += kThreads) scores[i] = 0u;
    for (int i = tid; i < T * kHistWords; i += kThreads) hist[i] = 0u;
    __syncthreads();
  }

  // The next kernel in the stream (sparse attention) may begin its prologue on idle SMs; it reads
  // nothing this kernel writes before this grid has completed.
  griddep_launch_dependents();

  // ---------------- select phase (cluster-uniform control flow)
  if (tid < T) {
    const int tt = tid;
    const int vis = max(0, min(pos0 + tt + 1, u_hi) - u_lo);  // visible positions of the unit
    ctl->need_total[tt] = tt < nt ? min(p.K, vis) : 0;
    ctl->radix[tt] = (tt < nt && vis > p.K) ? 1 : 0;
    ctl->need[tt] = ctl->need_total[tt];
    ctl->prefix[tt] = 0u;
  }
  __syncthreads();
  bool any_radix = false;
#pragma unroll
  for (int tt = 0; tt < T; ++tt) any_radix |= ctl->radix[tt] != 0;
  // Warp w owns the contiguous segment [w*seg, (w+1)*seg) of this CTA's positions (whole
  // multiples of 128: a lane reads 4 consecutive keys), so the compaction needs no block barrier.
  const int seg = ((nscan + kThreads / 32 - 1) / (kThreads / 32) + 127) / 128 * 128;
  const int e_lo = min(nscan, warp * seg), e_hi = min(nscan, e_lo + seg);

  // First radix pass (the epilogue built its histogram while the keys streamed): every CTA finds
  // the 11-bit bin that holds the K-th key and how many keys of the cluster fall into it.
  bool fast = false;
  if (any_radix) {
    cluster_sync();
    // every token of the group at once: its 2048 bins summed over the cluster, then one block
    // scan per token (sharing the barriers) finds the bin that holds its K-th key
    uint32_t cnt[T][8], sum[T], above[T];
#pragma unroll
    for (int tt = 0; tt < T; ++tt) {
#pragma unroll
      for (int k = 0; k < 8; ++k) cnt[tt][k] = 0u;
      if (tid < kHistThreads && ctl->radix[tt]) cluster_hist_sum(hist + tt * kHistWords + 4 * tid, p.C, cnt[tt]);
      sum[tt] = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k) sum[tt] += cnt[tt][k];
    }
    if (tid < T) {
      ctl->found_bin[tid] = 0;
      ctl->found_need[tid] = 1;
      ctl->cand_total[tid] = 0x7fffffff;
    }
    block_excl_suffix_multi<T>(sum, ctl->scan_t, above);
#pragma unroll
    for (int tt = 0; tt < T; ++tt) {
      if (!ctl->radix[tt]) continue;
      const uint32_t need = (uint32_t)ctl->need[tt];
      uint32_t run = above[tt];
#pragma unroll
      for (int k = 7; k >= 0; --k) {
        if (run < need && run + cnt[tt][k] >= need) {
          ctl->found_bin[tt] = 8 * tid + k;
          ctl->found_need[tt] = (int)(need - run);
          ctl->cand_total[tt] = (int)cnt[tt][k];
        }
        run += cnt[tt][k];
      }
    }
    __syncthreads();
    if (tid < T && ctl->radix[tid]) {
      ctl->prefix[tid] = (uint32_t)ctl->found_bin[tid] << 21;
      ctl->need[tid] = ctl->found_need[tid];
    }
    __syncthreads();
    // Candidate path when every threshold bin is small enough to gather into one CTA.
    const int cap = p.nstage * CF::kTileBytes / 2 / 8 / T;
    // a lane's candidate bits (4 per 128-key step of its warp segment) fit one 64-bit word
    fast = p.chunk <= 16 * 128 * (kThreads / 32);
#pragma unroll
    for (int tt = 0; tt < T; ++tt)
      if (ctl->radix[tt] && ctl->cand_total[tt] > cap) fast = false;  // uniform over the cluster
  }

  if (fast) {
    // ---- candidate path: one cluster barrier.  Every CTA reads how many keys each rank holds in
    // the threshold bin, so the cluster's candidate list has a known layout (rank order, then
    // position order) and every CTA pushes its candidates' keys straight into every other CTA's
    // copy of the list (asynchronous stores counted on the receiver's mbarrier); each CTA then
    // resolves the threshold and the per-rank counts from its full copy.
    const int cap = p.nstage * CF::kTileBytes / 2 / 8 / T;
    uint32_t* gk = reinterpret_cast<uint32_t*>(stage_base);  // [T][cap] the cluster's candidates
    // (a) candidates per rank in the threshold bin (first-pass histograms), list offsets, and the
    //     bytes the other ranks will store here: their candidates and their sure counts
    if (tid < T * p.C) {
      const int tt = tid / p.C, r = tid % p.C;
      int n = 0;
      if (ctl->radix[tt]) {
        const uint32_t bin = ctl->prefix[tt] >> 21;
        const uint32_t w = ld_cluster_u32(map_cluster(hist + tt * kHistWords + (bin >> 1), (uint32_t)r));
        n = (int)((w >> (16u * (bin & 1u))) & 0xffffu);
      }
      ctl->rn[tt][r] = n;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t bytes = 4u * T * (uint32_t)(p.C - 1);
      for (int tt = 0; tt < T; ++tt) {
        int o = 0;
        for (int r = 0; r < p.C; ++r) {
          ctl->roff[tt][r] = o;
          o += ctl->rn[tt][r];
          if (r != rank) bytes += 4u * (uint32_t)ctl->rn[tt][r];
        }
        ctl->cand_total[tt] = o;  // equals the histogram's count of the bin
      }
      // (a phase may count stored bytes before this arrival sets how many to expect)
      mbar_arrive_expect_tx(&ctl->cand_bar, bytes);
    }
    // (b) per warp segment: keys certainly selected ("sure": above the threshold bin, or every
    //     visible key of a token that sees fewer than K positions) are counted, keys in the
    //     threshold bin marked (bit 4*step + k of the lane's word) and counted per lane
    uint64_t cbits[4];
    int lane_base[4];
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      cbits[tt] = 0ull;
      lane_base[tt] = 0;
    }
    {
      // the tokens of the group scan the warp's segment together
      bool rdx[T];
      uint32_t b0[T], sure[T];
      uint64_t bits[T];
#pragma unroll
      for (int tt = 0; tt < T; ++tt) {
        rdx[tt] = ctl->radix[tt] != 0;
        b0[tt] = ctl->prefix[tt] >> 21;
        sure[tt] = 0u;
        bits[tt] = 0ull;
      }
#pragma unroll 2
      for (int e = e_lo + 4 * lane, it = 0; e < e_hi; e += 128, ++it) {
#pragma unroll
        for (int tt = 0; tt < T; ++tt) {
          const uint4 v = *reinterpret_cast<const uint4*>(scores + tt * p.chunk + e);
          const uint32_t us[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            sure[tt] += rdx[tt] ? ((us[k] >> 21) > b0[tt]) : (us[k] != 0u);
            if (rdx[tt] && us[k] != 0u && (us[k] >> 21) == b0[tt]) bits[tt] |= 1ull << (4 * it + k);
          }
        }
      }
      uint32_t mine[T], inc[T];
#pragma unroll
      for (int tt = 0; tt < T; ++tt) inc[tt] = mine[tt] = (uint32_t)__popcll(bits[tt]);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int tt = 0; tt < T; ++tt) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, inc[tt], o);
          if (lane >= o) inc[tt] += y;
        }
      }
#pragma unroll
      for (int tt = 0; tt < T; ++tt) {
        cbits[tt] = bits[tt];
        lane_base[tt] = (int)(inc[tt] - mine[tt]);
        const uint32_t sr = __reduce_add_sync(0xffffffffu, sure[tt]);
        const uint32_t cand = __shfl_sync(0xffffffffu, inc[tt], 31);
        if (lane == 0) {
          ctl->wgt[tt][warp] = (int)sr;
          ctl->wcnd[tt][warp] = (int)cand;
        }
      }
    }
    __syncthreads();
    // (c) each lane stores its candidates' keys at their place in the cluster's list (this rank's
    //     range, warps in order, lane-major within a warp) here and in every other CTA, and the
    //     CTA's sure counts go to every other CTA
    if (tid < T) {
      int g = 0;
      for (int w = 0; w < kThreads / 32; ++w) g += ctl->wgt[tid][w];
      ctl->rsure[tid][rank] = g;
      for (int r = 0; r < p.C; ++r)
        if (r != rank)
          st_async_b32(map_cluster(&ctl->rsure[tid][rank], (uint32_t)r), (uint32_t)g,
                       map_cluster(&ctl->cand_bar, (uint32_t)r));
    }
#pragma unroll
    for (int tt = 0; tt < T; ++tt) {
      if (!ctl->radix[tt]) continue;
      const uint32_t* sc = scores + tt * p.chunk;
      int slot = ctl->roff[tt][rank] + lane_base[tt];
      for (int w = 0; w < warp; ++w) slot += ctl->wcnd[tt][w];
      uint64_t bits = cbits[tt];
      while (bits) {
        const int bit = __ffsll((long long)bits) - 1;
        bits &= bits - 1ull;
        const uint32_t key = sc[e_lo + 128 * (bit >> 2) + 4 * lane + (bit & 3)];
        gk[tt * cap + slot] = key;
        for (int r = 0; r < p.C; ++r)
          if (r != rank)
            st_async_b32(map_cluster(gk + tt * cap + slot, (uint32_t)r), key,
                         map_cluster(&ctl->cand_bar, (uint32_t)r));
        ++slot;
      }
    }
    cluster_arrive();  // this CTA has finished reading and storing into the other CTAs' memory
    {
      const bool ok = mbar_wait<true>(&ctl->cand_bar, 0u, abort, p.status);
      (void)ok;  // after a timeout the candidates are incomplete: the result is unspecified
    }
    __syncthreads();  // every thread's own stores into gk are visible too
    // (d) the remaining 21 bits among the gathered candidates, locally (no cluster barrier;
    //     every peer has finished reading this CTA's histogram before sending its candidates):
    // a histogram of bits 20..10, then the last 10 bits directly among the few candidates that
    // share the 22-bit prefix (a histogram again when there are more than kFew)
    constexpr int kFew = 64;
    uint32_t* few = hist + kHistWords;  // scratch beside the local histogram
#pragma unroll 1
    for (int tt = 0; tt < T; ++tt) {
      if (!ctl->radix[tt]) continue;
      const int n = ctl->cand_total[tt];
      const uint32_t* G = gk + tt * cap;
      uint32_t* h = hist;
      {  // bits 20..10
        const uint32_t pref = ctl->prefix[tt];
        for (int i = tid; i < kHistWords; i += kThreads) h[i] = 0u;
        if (tid == 0) ctl->few_cnt = 0;
        __syncthreads();
        for (int i = tid; i < n; i += kThreads) {
          const uint32_t u = G[i];
          if ((u & 0xffe00000u) == pref) {
            const uint32_t bin = (u >> 10) & 2047u;
            atomicAdd(&h[bin >> 1], 1u << ((bin & 1u) * 16u));
          }
        }
        __syncthreads();
        find_bin_local(h, (uint32_t)ctl->need[tt], tt, ctl);
        if (tid == 0) {
          ctl->prefix[tt] |= (uint32_t)ctl->found_bin[tt] << 10;
          ctl->need[tt] = ctl->found_need[tt];
        }
        __syncthreads();
      }
      const uint32_t pref = ctl->prefix[tt];
      for (int i = tid; i < n; i += kThreads) {
        const uint32_t u = G[i];
        if ((u & 0xfffffc00u) == pref) {
          const int slot = atomicAdd(&ctl->few_cnt, 1);
          if (slot < kFew) few[slot] = u;
        }
      }
      __syncthreads();
      const int m = ctl->few_cnt;  // uniform over the block
      if (m <= kFew) {
        // the need-th largest of the m keys: the key with (greater) < need <= (greater or equal)
        if (tid < m) {
          const uint32_t v = few[tid];
          int gt = 0, ge = 0;
          for (int j = 0; j < m; ++j) {
            gt += few[j] > v;
            ge += few[j] >= v;
          }
          const int need = ctl->need[tt];
          if (gt < need && need <= ge) {  // equal keys write equal values
            ctl->found_bin[tt] = (int)v;
            ctl->found_need[tt] = need - gt;
          }
        }
        __syncthreads();
        if (tid == 0) {
          ctl->prefix[tt] = (uint32_t)ctl->found_bin[tt];
          ctl->need[tt] = ctl->found_need[tt];
        }
        __syncthreads();
      } else {  // bits 9..0 by histogram
        for (int i = tid; i < kHistWords; i += kThreads) h[i] = 0u;
        __syncthreads();
        for (int i = tid; i < n; i += kThreads) {
          const uint32_t u = G[i];
          if ((u & 0xfffffc00u) == pref) {
            const uint32_t bin = u & 1023u;
            atomicAdd(&h[bin >> 1], 1u << ((bin & 1u) * 16u));
          }
        }
        __syncthreads();
        find_bin_local(h, (uint32_t)ctl->need[tt], tt, ctl);
        if (tid == 0) {
          ctl->prefix[tt] |= (uint32_t)ctl->found_bin[tt];
          ctl->need[tt] = ctl->found_need[tt];
        }
        __syncthreads();
      }
    }
    // (e) candidates above / at the threshold per rank (its range of the list), and per warp of
    //     this CTA (its range within this rank's)
    if (tid < T * p.C) {
      ctl->rgt[tid / p.C][tid % p.C] = 0;
      ctl->req[tid / p.C][tid % p.C] = 0;
    }
    __syncthreads();
#pragma unroll 1
    for (int tt = 0; tt < T; ++tt) {
      if (!ctl->radix[tt]) continue;  // uniform over the block
      const uint32_t thr = ctl->prefix[tt];
      const uint32_t* G = gk + tt * cap;
      for (int r = warp; r < p.C; r += kThreads / 32) {
        const int r0 = ctl->roff[tt][r], r1 = r0 + ctl->rn[tt][r];
        uint32_t ng = 0, ne = 0;
        for (int i = r0 + lane; i < r1; i += 32) {
          ng += G[i] > thr;
          ne += G[i] == thr;
        }
        ng = __reduce_add_sync(0xffffffffu, ng);
        ne = __reduce_add_sync(0xffffffffu, ne);
        if (lane == 0) {
          ctl->rgt[tt][r] = (int)ng;
          ctl->req[tt][r] = (int)ne;
        }
      }
      {
        int w0 = ctl->roff[tt][rank];
        for (int w = 0; w < warp; ++w) w0 += ctl->wcnd[tt][w];
        const int w1 = w0 + ctl->wcnd[tt][warp];
        uint32_t ng = 0, ne = 0;
        for (int i = w0 + lane; i < w1; i += 32) {
          ng += G[i] > thr;
          ne += G[i] == thr;
        }
        ng = __reduce_add_sync(0xffffffffu, ng);
        ne = __reduce_add_sync(0xffffffffu, ne);
        if (lane == 0) {
          ctl->wgt[tt][warp] += (int)ng;  // sure keys + candidates above the threshold
          ctl->weq[tt][warp] = (int)ne;
        }
      }
    }
    if (tid < T * (kThreads / 32)) {
      const int tt = tid / (kThreads / 32), w = tid % (kThreads / 32);
      if (!ctl->radix[tt]) ctl->weq[tt][w] = 0;
    }
    __syncthreads();
    if (tid < T) {
      const int tt = tid;
      const int need_eq = ctl->radix[tt] ? ctl->need[tt] : 0;
      int eq_before = 0, off = 0, my_quota = 0;
      for (int r = 0; r < p.C; ++r) {
        const int gt_r = ctl->rsure[tt][r] + ctl->rgt[tt][r];
        const int eq_r = ctl->req[tt][r];
        const int quota_r = max(0, min(eq_r, need_eq - eq_before));
        if (r < rank) off += gt_r + quota_r;
        if (r == rank) my_quota = quota_r;
        eq_before += eq_r;
      }
      ctl->offset[tt] = off;
      ctl->quota[tt] = my_quota;
    }
    __syncthreads();
  } else {
    // ---- general path: radix passes 2 and 3 over every key, cluster-wide
    if (any_radix) {
#pragma unroll 1
      for (int pass = 1; pass < 3; ++pass) {
        const int shift = pass == 1 ? 10 : 0;
        const int nbits = pass == 2 ? 10 : 11;
        const uint32_t bmask = (1u << nbits) - 1u;
        const uint32_t pmask = 0xffffffffu << (shift + nbits);
        uint32_t* hb = hist + (pass & 1) * T * kHistWords;
        for (int i = tid; i < T * kHistWords; i += kThreads) hb[i] = 0u;
        __syncthreads();
#pragma unroll 1
        for (int tt = 0; tt < T; ++tt) {
          if (!ctl->radix[tt]) continue;
          const uint32_t pref = ctl->prefix[tt];
          const uint4* sc4 = reinterpret_cast<const uint4*>(scores + tt * p.chunk);
          uint32_t* h = hb + tt * kHistWords;
#pragma unroll 4
          for (int e4 = tid; e4 < nscan / 4; e4 += kThreads) {
            const uint4 v = sc4[e4];
            const uint32_t us[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t u = us[k];
              if (u != 0u && (u & pmask) == pref) {
                const uint32_t bin = (u >> shift) & bmask;
                atomicAdd(&h[bin >> 1], 1u << ((bin & 1u) * 16u));
              }
            }
          }
        }
        cluster_sync();
#pragma unroll 1
        for (int tt = 0; tt < T; ++tt) {
          if (!ctl->radix[tt]) continue;  // uniform over the block
          uint32_t cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          if (tid < kHistThreads) {
            const uint32_t* h = hb + tt * kHistWords + 4 * tid;
            cluster_hist_sum(h, p.C, cnt);
          }
          uint32_t sum = 0;
#pragma unroll
          for (int k = 0; k < 8; ++k) sum += cnt[k];
          if (tid == 0) {
            ctl->found_bin[tt] = 0;
            ctl->found_need[tt] = 1;
          }
          const uint32_t above = block_excl_suffix(sum, ctl->scan);
          const uint32_t need = (uint32_t)ctl->need[tt];
          uint32_t run = above;
#pragma unroll
          for (int k = 7; k >= 0; --k) {
            if (run < need && run + cnt[k] >= need) {
              ctl->found_bin[tt] = 8 * tid + k;
              ctl->found_need[tt] = (int)(need - run);
            }
            run += cnt[k];
          }
          __syncthreads();
          if (tid == 0) {
            ctl->prefix[tt] |= (uint32_t)ctl->found_bin[tt] << shift;
            ctl->need[tt] = ctl->found_need[tt];
          }
          __syncthreads();
        }
      }
    }
    // counts above / at the threshold, per warp segment and per CTA
#pragma unroll 1
    for (int tt = 0; tt < T; ++tt) {
      const uint32_t thr = ctl->radix[tt] ? ctl->prefix[tt] : 0u;
      const uint32_t* sc = scores + tt * p.chunk;
      uint32_t gt = 0, eq = 0;
#pragma unroll 4
      for (int e = e_lo + 4 * lane; e < e_hi; e += 128) {
        const uint4 v = *reinterpret_cast<const uint4*>(sc + e);
        const uint32_t us[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          gt += us[k] > thr;
          eq += (us[k] == thr && us[k] != 0u);
        }
      }
      gt = __reduce_add_sync(0xffffffffu, gt);
      eq = __reduce_add_sync(0xffffffffu, eq);
      if (lane == 0) {
        ctl->wgt[tt][warp] = (int)gt;
        ctl->weq[tt][warp] = (int)eq;
      }
    }
    __syncthreads();
    if (tid < T) {
      int g = 0, q = 0;
      for (int w = 0; w < kThreads / 32; ++w) {
        g += ctl->wgt[tid][w];
        q += ctl->weq[tid][w];
      }
      ctl->cnt_gt[tid] = g;
      ctl->cnt_eq[tid] = q;
    }
    cluster_sync();
    if (tid < T) {
      const int tt = tid;
      const int need_eq = ctl->radix[tt] ? ctl->need[tt] : 0;
      int eq_before = 0, off = 0, my_quota = 0;
      for (int r = 0; r < p.C; ++r) {
        const int gt_r = (int)ld_cluster_u32(map_cluster(&ctl->cnt_gt[tt], (uint32_t)r));
        const int eq_r = (int)ld_cluster_u32(map_cluster(&ctl->cnt_eq[tt], (uint32_t)r));
        const int quota_r = max(0, min(eq_r, need_eq - eq_before));
        if (r < rank) off += gt_r + quota_r;
        if (r == rank) my_quota = quota_r;
        eq_before += eq_r;
      }
      ctl->offset[tt] = off;
      ctl->quota[tt] = my_quota;
    }
    __syncthreads();
  }

  // ascending-position compaction: ties at the threshold go to the lowest positions.  A warp
  // stages its selected positions in place at the front of its own segment of the key array
  // (never ahead of what it has read), then writes them out with coalesced stores.  The tokens
  // of a group go through each 512-key batch together, so their latency chains overlap.
  {
    int off_t[T], ties_t[T], need_t[T], eqr_t[T], selr_t[T];
    uint32_t thr_t[T];
    bool rdx_t[T];
    int* out_t[T];
    float* osc_t[T];
#pragma unroll
    for (int tt = 0; tt < T; ++tt) {
      off_t[tt] = ties_t[tt] = need_t[tt] = eqr_t[tt] = selr_t[tt] = 0;
      thr_t[tt] = 0u;
      rdx_t[tt] = false;
      out_t[tt] = nullptr;
      osc_t[tt] = nullptr;
      if (tt < nt) {
        rdx_t[tt] = ctl->radix[tt] != 0;
        thr_t[tt] = rdx_t[tt] ? ctl->prefix[tt] : 0u;
        need_t[tt] = ctl->need_total[tt];
        int eq_before = 0, off = ctl->offset[tt];
        for (int w = 0; w < warp; ++w) {
          const int ties_w = max(0, min(ctl->weq[tt][w], ctl->quota[tt] - eq_before));
          off += ctl->wgt[tt][w] + ties_w;
          eq_before += ctl->weq[tt][w];
        }
        off_t[tt] = off;
        ties_t[tt] = max(0, min(ctl->weq[tt][warp], ctl->quota[tt] - eq_before));
        const size_t slot_u = ((size_t)(b * p.groups + g) * p.units + unit) * T + tt;
        out_t[tt] = direct ? p.out_idx + (size_t)(t0 + tt) * p.K : p.cand_idx + slot_u * p.K;
        osc_t[tt] = direct ? (p.out_score ? p.out_score + (size_t)(t0 + tt) * p.K : nullptr)
                           : p.cand_score + slot_u * p.K;
      }
    }
    // batches of four 128-key groups: lane holds keys 4*lane..4*lane+3 of each group
#pragma unroll 1
    for (int eb = e_lo; eb < e_hi; eb += 512) {
      uint32_t key[T][16], take[T], feq[T], tinc[T], tcnt[T];
#pragma unroll
      for (int tt = 0; tt < T; ++tt) {
        take[tt] = feq[tt] = 0u;
        if (tt < nt) {
          const uint32_t* sc = scores + tt * p.chunk;
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (eb + 128 * gg < e_hi) v = *reinterpret_cast<const uint4*>(sc + eb + 128 * gg + 4 * lane);
            key[tt][4 * gg + 0] = v.x; key[tt][4 * gg + 1] = v.y;
            key[tt][4 * gg + 2] = v.z; key[tt][4 * gg + 3] = v.w;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t u = key[tt][4 * gg + k];
              if (u > thr_t[tt]) take[tt] |= 1u << (4 * gg + k);
              if (rdx_t[tt] && u == thr_t[tt] && u != 0u) feq[tt] |= 1u << (4 * gg + k);
            }
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < T; ++tt) {
        if (tt < nt && __any_sync(0xffffffffu, feq[tt] != 0u)) {
          // keys equal to the threshold: this warp takes the first ties_t of them
          const uint32_t ecnt = nibble_counts(feq[tt]);
          const uint32_t einc = warp_incl_scan(ecnt);
          const uint32_t etot = __shfl_sync(0xffffffffu, einc, 31);
          const uint32_t eexc = einc - ecnt;
          int ebase = eqr_t[tt];
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
            int seen = ebase + (int)((eexc >> (8 * gg)) & 0xffu);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if ((feq[tt] >> (4 * gg + k)) & 1u) {
                if (seen < ties_t[tt]) take[tt] |= 1u << (4 * gg + k);
                ++seen;
              }
            ebase += (int)((etot >> (8 * gg)) & 0xffu);
          }
          eqr_t[tt] = ebase;
        }
      }
      // the tokens' packed warp scans, step by step
#pragma unroll
      for (int tt = 0; tt < T; ++tt) tinc[tt] = tcnt[tt] = nibble_counts(take[tt]);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int tt = 0; tt < T; ++tt) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, tinc[tt], o);
          if (lane >= o) tinc[tt] += y;
        }
      }
#pragma unroll
      for (int tt = 0; tt < T; ++tt) {
        if (tt >= nt) continue;
        uint32_t* sc = scores + tt * p.chunk;
        const uint32_t ttot = __shfl_sync(0xffffffffu, tinc[tt], 31);
        const uint32_t texc = tinc[tt] - tcnt[tt];
        // every lane's keys of the batch are in registers (the scan above), and the staged
        // count never exceeds the keys read so far: the writes land on keys already consumed
        int base = selr_t[tt];
        if (osc_t[tt] == nullptr) {
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
            int slot = e_lo + base + (int)((texc >> (8 * gg)) & 0xffu);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if ((take[tt] >> (4 * gg + k)) & 1u) sc[slot++] = (uint32_t)(lo + eb + 128 * gg + 4 * lane + k);
            base += (int)((ttot >> (8 * gg)) & 0xffu);
          }
        } else {  // also the score of each selected position (uncoalesced; optional output)
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
            int slot = e_lo + base + (int)((texc >> (8 * gg)) & 0xffu);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if ((take[tt] >> (4 * gg + k)) & 1u) {
                if (off_t[tt] + (slot - e_lo) < need_t[tt])
                  osc_t[tt][off_t[tt] + (slot - e_lo)] = key_score(key[tt][4 * gg + k]);
                sc[slot++] = (uint32_t)(lo + eb + 128 * gg + 4 * lane + k);
              }
            base += (int)((ttot >> (8 * gg)) & 0xffu);
          }
        }
        selr_t[tt] = base;
      }
    }
    __syncwarp();
#pragma unroll
    for (int tt = 0; tt < T; ++tt) {
      if (tt >= nt) continue;
      const uint32_t* sc = scores + tt * p.chunk;
      for (int j = lane; j < selr_t[tt]; j += 32) {
        if (off_t[tt] + j < need_t[tt])
          out_t[tt][off_t[tt] + j] = (int)sc[e_lo + j];
        else
          report(p.status, kStatusDeviceCheck);
      }
      if (rank == 0) {
        for (int r = need_t[tt] + tid; r < p.K; r += kThreads) {
          out_t[tt][r] = -1;
          if (osc_t[tt]) osc_t[tt][r] = -INFINITY;
        }
        if (direct && tid == 0 && p.out_cnt) p.out_cnt[t0 + tt] = need_t[tt];
      }
    }
  }
  // peers may still be reading this CTA's counters / candidates
  if (fast)
    cluster_wait();
  else
    cluster_sync();
}

// Unit plan: one CTA lists the (sequence, unit) items of a launch with position units, in the
// order of decreasing unit length (ties by sequence), so the longest work starts first; clusters
// then read their item from the list.  A sequence of L positions has ceil(L / span) units of
// ceil(L / units) positions.
__global__ void __launch_bounds__(256) unit_plan_kernel(const int* seq_lens, int B, int span,
                                                        int units, int* items) {
  __shared__ int ulen[kMaxUnitSeqs], ucnt[kMaxUnitSeqs];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < B) {
    const int L = max(0, seq_lens[tid]);
    // (a length beyond units * span is reported by the indexer; the list stays in bounds)
    const int nu = min(units, max(1, (L + span - 1) / span));
    ulen[tid] = (L + nu - 1) / nu;
    ucnt[tid] = nu;
  }
  __syncthreads();
  // a warp per sequence: its lanes count the units of the sequences ordered before it
  for (int i = warp; i < B; i += 8) {
    const int li = ulen[i];
    int start = 0;
    for (int j = lane; j < B; j += 32)
      start += (ulen[j] > li || (ulen[j] == li && j < i)) ? ucnt[j] : 0;
    start = (int)__reduce_add_sync(0xffffffffu, (uint32_t)start);
    if (lane < ucnt[i]) items[1 + start + lane] = (i << 8) | lane;
  }
  if (warp == 0) {
    int total = 0;
    for (int j = lane; j < B; j += 32) total += ucnt[j];
    total = (int)__reduce_add_sync(0xffffffffu, (uint32_t)total);
    if (lane == 0) items[0] = total;
  }
}

// ---------------------------------------------------------------- host side

// Upper bound of the position units per sequence (1: a cluster covers a whole sequence).  Units
// are used for groups of at most two tokens (decode, speculative pairs) whose sequences may be
// longer than kUnitSpan, as long as the merge can hold every unit's candidates.
static int unit_bound(const dsa_li_args& a) {
  // (the longest-first order of the units is derived in every CTA: at most kMaxUnitSeqs)
  if (a.max_q_per_seq > 2 || a.max_seq_len <= kUnitSpan || a.B > kMaxUnitSeqs) return 1;
  const int u = (a.max_seq_len + kUnitSpan - 1) / kUnitSpan;
  return (long long)u * a.K <= kMaxUnitCand ? u : 1;
}

static size_t unit_workspace_bytes(const dsa_li_args& a) {
  const int ub = unit_bound(a);
  if (ub <= 1) return 0;
  const int T = a.max_q_per_seq <= 1 ? 1 : 2;
  const int groups = (a.max_q_per_seq + T - 1) / T;
  const size_t slots = (size_t)a.B * groups * ub * T;
  return 2 * ((slots * a.K * 4 + 255) / 256 * 256) + ((1 + (size_t)a.B * ub) * 4 + 255) / 256 * 256;
}

template <int D_I, bool FP8, int H_I, int T, bool MX = false>
static dsa_status launch_impl(const dsa_li_args& a, cudaStream_t stream, std::string& err) {
  using CF = Cfg<D_I, FP8, H_I, T, MX>;
  DeviceInfo dev;
  if (!device_info(dev, err)) return DSA_ERR_CUDA;
  const int groups = (a.max_q_per_seq + T - 1) / T;
  const int maxL = std::max(a.max_seq_len, 1);
  // With units, a cluster is planned for kUnitSpan positions and a sequence takes one cluster
  // per unit; otherwise for the longest sequence.
  const int ub = T <= 2 ? unit_bound(a) : 1;
  const int planL = ub > 1 ? kUnitSpan : maxL;

  auto kern = li_topk_kernel<D_I, FP8, H_I, T, MX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.smem_optin);
  if (e != cudaSuccess) return cuda_fail(e, "li_topk: set shared memory size", err);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return cuda_fail(e, "li_topk: allow cluster > 8", err);

  // Pick ring depth, cluster size and chunk with the occupancy API: how many clusters of each
  // shape the GPU co-schedules decides the number of waves; within a wave the time is set by the
  // HBM share of the resident CTAs, by how many bytes one SM keeps in flight, and by the
  // select phase (which scans each CTA's chunk and does not overlap the stream).
  struct Choice { int ns, c, chunk, smem; };
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int>, Choice> memo;
  const auto key = std::make_tuple(dev.device, maxL, a.B * groups, ub);
  Choice best{0, 0, 0, 0};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find(key);
    if (it != memo.end()) best = it->second;
  }
  if (!best.c) {
    double best_est = 1e300;
    for (int ns = 8; ns >= 2; --ns) {
      for (int c = 1; c <= kMaxCluster; ++c) {
        const int chunk = ((planL + c - 1) / c + kTileKeys - 1) / kTileKeys * kTileKeys;
        if (chunk > 65535 || (long long)chunk * c < planL) continue;
        if (ub > 1 && chunk * c != kUnitSpan) continue;  // units of exactly kUnitSpan positions
        const long long units = ub > 1 ? (maxL + (long long)c * chunk - 1) / ((long long)c * chunk) : 1;
        const long long clusters = (long long)a.B * groups * units;
        const Layout lay(ns, CF::kTileBytes, CF::kQBytes, T, H_I, chunk);
        const int smem = lay.total + 1024;
        if (smem > dev.smem_optin) continue;
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3((unsigned)(c * clusters));
        q.blockDim = dim3(kThreads);
        q.dynamicSmemBytes = (size_t)smem;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)c;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        q.attrs = at;
        q.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, kern, &q) != cudaSuccess || active <= 0) {
          cudaGetLastError();
          continue;
        }
        const long long waves = (clusters + active - 1) / active;
        const long long resident = std::min<long long>(clusters, active) * c;
        const double per_sm = std::ceil((double)resident / dev.sm_count);
        const double bytes_cta = (double)chunk * CF::kRowBytes;
        const double hbm = 6.4e12, latency = 1.3e-6, sm_cap = 160e9;
        const double sm_bw = std::min(sm_cap, per_sm * ns * CF::kTileBytes / latency);
        const double t_stream = std::max(resident * bytes_cta / hbm, per_sm * bytes_cta / sm_bw);
        const double t_select = 4e-6 + (double)chunk * T * 1.5e-9;
        const double est = (double)waves * (t_stream + t_select);
        if (est < best_est * 0.995) {
          best_est = est;
          best = Choice{ns, c, chunk, smem};
        }
      }
    }
    if (!best.c) {
      err = "li_topk: no (ring depth, cluster size) fits for max_seq_len " + std::to_string(a.max_seq_len);
      return DSA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(mu);
    memo[key] = best;
  }
  const int best_ns = best.ns, best_c = best.c, best_chunk = best.chunk, best_smem = best.smem;
  const int units = ub > 1 ? (maxL + best_c * best_chunk - 1) / (best_c * best_chunk) : 1;
  UnitMergeArgs um{};
  int* items = nullptr;
  if (units > 1) {
    const size_t slots = (size_t)a.B * groups * units * T;
    const size_t half = (slots * a.K * 4 + 255) / 256 * 256;
    const size_t need = 2 * half + ((1 + (size_t)a.B * units) * 4 + 255) / 256 * 256;
    if (a.workspace == nullptr || a.workspace_bytes < need) {
      err = "li_topk: workspace of " + std::to_string(need) + " bytes required (got " +
            std::to_string(a.workspace_bytes) + ")";
      return DSA_ERR_INVALID_ARG;
    }
    um.cand_idx = reinterpret_cast<int*>(a.workspace);
    um.cand_score = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(a.workspace) + half);
    items = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(a.workspace) + 2 * half);
    unit_plan_kernel<<<1, 256, 0, stream>>>(a.seq_lens, a.B, best_c * best_chunk, units, items);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "li_topk: unit plan launch", err);
  }

  CUtensorMap tm_k, tm_q;
  const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_tmap_2d(&tm_k, dt, a.k_pool, D_I, (uint64_t)a.num_pages * 64, CF::kRowBytes,
                      CF::kBoxW / CF::kElt, 64,
                      CF::kBoxW == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, err))
    return DSA_ERR_CUDA;
  if (!encode_tmap_2d(&tm_q, dt, a.q, D_I, (uint64_t)a.n_q * H_I, CF::kRowBytes, 128 / CF::kElt,
                      CF::kNCol, CU_TENSOR_MAP_SWIZZLE_128B, err))
    return DSA_ERR_CUDA;

  Params p;
  p.B = a.B;
  p.n_q = a.n_q;
  p.K = a.K;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.groups = groups;
  p.chunk = best_chunk;
  p.C = best_c;
  p.units = units;
  p.nstage = best_ns;
  p.w = a.w;
  p.q_scale = a.q_scale;
  p.k_scale = a.k_scale;
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.q_start = a.q_start;
  p.out_idx = a.out_idx;
  p.out_cnt = a.out_cnt;
  p.status = a.status;
  p.q_sf = a.q_sf;
  p.k_sf = a.k_sf;
  p.out_score = a.out_score;
  p.cand_idx = um.cand_idx;
  p.cand_score = um.cand_score;
  p.items = items;
#ifdef DSA_TEST_HOOKS
  p.stall = g_test_stall;
#endif

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(best_c * a.B * groups * units));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)best_smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)best_c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // with units: a programmatic dependent of the unit plan (waits for it before any read)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = units > 1 ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kern, tm_k, tm_q, p);
  if (e != cudaSuccess) return cuda_fail(e, "li_topk: launch", err);
  if (units > 1) {
    um.B = a.B;
    um.n_q = a.n_q;
    um.K = a.K;
    um.T = T;
    um.groups = groups;
    um.units = units;
    um.span = best_c * best_chunk;
    um.max_pages = a.max_pages;
    um.seq_lens = a.seq_lens;
    um.q_start = a.q_start;
    um.out_idx = a.out_idx;
    um.out_cnt = a.out_cnt;
    um.out_score = a.out_score;
    return launch_unit_merge(um, stream, err);
  }
  return DSA_OK;
}

}  // namespace li

size_t li_workspace_bytes(const dsa_li_args& a) { return li::unit_workspace_bytes(a); }

static dsa_status launch_li_topk_T(const dsa_li_args& a, int T, cudaStream_t stream, std::string& err);

dsa_status launch_li_topk(const dsa_li_args& a, cudaStream_t stream, std::string& err) {
  // Tokens per cluster: all new tokens of a sequence up to 4 (4 x 64 heads = the widest MMA N);
  // if a group of 4 does not fit shared memory at this context length, groups of 2.
  int T = a.max_q_per_seq <= 1 ? 1 : (a.max_q_per_seq <= 2 ? 2 : 4);
  dsa_status s = launch_li_topk_T(a, T, stream, err);
  if (s == DSA_ERR_UNSUPPORTED && T == 4) s = launch_li_topk_T(a, 2, stream, err);
  return s;
}

static dsa_status launch_li_topk_T(const dsa_li_args& a, int T, cudaStream_t stream, std::string& err) {
  const bool fp8 = a.dtype == DSA_FP8_E4M3;
  const bool mx = a.dtype == DSA_MXFP8_E4M3;
  if (a.H_I == 64 && a.d_I == 128) {
    if (mx) {  // at most 2 tokens per group: the scale cells need tensor memory beside 2 x 128 columns
      if (T == 1) return li::launch_impl<128, true, 64, 1, true>(a, stream, err);
      return li::launch_impl<128, true, 64, 2, true>(a, stream, err);
    }
    if (fp8) {
      if (T == 1) return li::launch_impl<128, true, 64, 1>(a, stream, err);
      if (T == 2) return li::launch_impl<128, true, 64, 2>(a, stream, err);
      return li::launch_impl<128, true, 64, 4>(a, stream, err);
    }
    if (T == 1) return li::launch_impl<128, false, 64, 1>(a, stream, err);
    if (T == 2) return li::launch_impl<128, false, 64, 2>(a, stream, err);
    return li::launch_impl<128, false, 64, 4>(a, stream, err);
  }
  if (a.H_I == 8 && a.d_I == 64 && !fp8 && !mx) {
    if (T == 1) return li::launch_impl<64, false, 8, 1>(a, stream, err);
    if (T == 2) return li::launch_impl<64, false, 8, 2>(a, stream, err);
    return li::launch_impl<64, false, 8, 4>(a, stream, err);
  }
  err = "li_topk: unsupported (H_I, d_I, dtype) = (" + std::to_string(a.H_I) + ", " +
        std::to_string(a.d_I) + ", " + (mx ? "mxfp8" : fp8 ? "fp8" : "bf16") + ")";
  return DSA_ERR_UNSUPPORTED;
}

}  // namespace dsa
