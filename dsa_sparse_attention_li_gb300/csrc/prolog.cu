// prolog.cu -- Indexer Prolog: the indexer's input preparation for the new tokens, in one launch.
//
// Method: "Inference Optimization for Kimi K3.1 Pro: Decoding Architecture Evolution and Systems
// Engineering Practices", section 3 (Indexer Prolog: the Q projection, the K normalisation of the
// input activations, and the Q quantisation with the head-weight projection are prepared
// concurrently and meet before the indexer) and section 4 (the indexer's MXFP8 path, 32-element
// groups); "Day0 Inference Adaptation for Next-Gen LLMs ... CANN", section 3.3 (projections in
// BF16, indexer inputs quantised per group of 32).  Per new token t at position p:
//   q[t] = W_q . xq[t]                        -> MXFP8 (codes + E8M0 group scales) or bf16
//   k[t] = LayerNorm(W_k . x[t]) * g + b      -> MXFP8 or bf16, written to the paged key cache
//   w[t] = w_scale * (W_w . x[t])             -> fp32 head weights
//
// GB300 design.  The pages' three streams become three CTA roles of one grid.  Each CTA computes
// one [128 output features x N tokens] tile of one projection over a slice of the input
// dimension: warp 0 streams 128-byte-wide chunks of the weight rows and of the activations with
// TMA into a 4-stage ring, warp 1 issues tcgen05.mma (bf16, fp32 accumulator in tensor memory).
// The slices of a tile are CTAs of one thread-block cluster (a cluster holds S / P tiles of P
// slices each), and the cluster's 2 S warpgroups share the tiles' rows (one row = one token's 128
// features, thread f holding feature f).  Every CTA reads its fp32 partial tile out of tensor
// memory and pushes each row with st.async into the shared memory of the warpgroup that finishes
// it (completion counted in bytes on that warpgroup's mbarrier, armed before the stream starts);
// the warpgroup adds the P partial rows in slice order -- deterministic -- and applies the
// epilogue:
//   Q tiles (one per index head: 128 features = d_I): one warp holds one 32-feature group, so
//     the MX shared exponent is a warp max; e4m3 rounding to nearest even with saturation;
//   K tiles: LayerNorm over the 128 features (warpgroup reduction), quantisation, and the store
//     of the key row at the token's physical cache row (page table, resolved while the
//     projection streams);
//   W tiles: the head weights (H_I = 64 rows of the tile).
// A split cluster barrier orders the barriers' initialisation before the first remote store and
// keeps every CTA resident until the cluster's stores have been issued.
#include <cuda_fp8.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace prolog {

constexpr int kThreads = 256;           // two warpgroups: each owns one lane quadrant per warp
constexpr int kGroupTok = 8;            // tokens per tensor-memory load (8 columns)
constexpr int kChunk = 64;                // input elements per ring step (a 128-byte bf16 row)
constexpr int kStages = 4;
constexpr int kATileBytes = 128 * 128;    // 128 weight rows x 128 B
constexpr int kTokBlock = 16;             // tokens per tensor-memory pass (8 per warpgroup)
constexpr int kMaxCluster = 16;           // CTAs per cluster (beyond 8: non-portable size)
constexpr int kRowBatch = 4;              // rows a warpgroup finishes together
constexpr int kMaxOwnRows = 64;           // rows of one warpgroup at most: 128 tokens / 2 warpgroups

struct Params {
  int n_q, B, H_I, mx;
  int ntok_q, ntok_kw;          // tokens per tile (MMA N, a power of two) of the Q / the K, W tiles
  int tiles_q, tiles_kw;        // token tiles of each
  int stage_max;                // ring stage bytes of the widest role
  int S;                        // CTAs per cluster
  int P_q, P_kw;                // slices per tile of each role (divisors of S)
  int units_q, units_k;         // Q tiles = 64 heads x tiles_q (unit = tile * 64 + head); K tiles
                                // = W tiles = tiles_kw
  int ctas_q, ctas_k;           // grid: [K CTAs][W CTAs][Q CTAs], each a multiple of S
  int chunks_q, chunks_kw;      // input chunks of the Q and of the K / W projections
  int recv_bytes;               // received partial rows [2][rows per warpgroup][P][128] fp32
  int max_pages, num_pages;
  float ln_eps, w_scale;
  const float* ln_gamma;
  const float* ln_beta;
  const int* page_table;
  const int* seq_lens;
  const int* q_start;
  uint8_t* q_out;
  uint8_t* q_sf;
  float* w_out;
  uint8_t* k_pool;
  uint8_t* k_sf;
  int* status;
};

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t done;
  uint64_t recv[2];                        // per warpgroup: its rows' partials have arrived
  uint32_t tmem_base;
  int abort;
  float red[2][kThreads / 32][kRowBatch];  // LayerNorm sums: [sum | squares][warp][row]
  long long krow[2][kMaxOwnRows];          // K rows of each warpgroup: key-cache row (-1: none)
};

DSA_DEV int find_seq(const int* q_start, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {  // largest b with q_start[b] <= t
    const int mid = (lo + hi + 1) >> 1;
    if (q_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

DSA_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// MX quantisation of one 32-value group held one value per lane: returns this lane's e4m3 code
// and (through sf) the group's E8M0 scale byte.  Shared exponent floor(log2 amax) - 8, clamped
// to [-127, 127] (0 for an all-zero group); elements rounded to nearest even, saturated at 448.
DSA_DEV uint8_t mx_quant_lane(float v, uint8_t* sf) {
  const uint32_t a = __reduce_max_sync(0xffffffffu, __float_as_uint(v) & 0x7fffffffu);  // |amax|
  // floor(log2 amax) is the biased exponent field - 127 for a normal amax; a subnormal amax
  // clamps to -127 either way
  const int e = a == 0u ? 0 : min(127, max(-127, (int)(a >> 23) - 127 - 8));
  *sf = (uint8_t)(e + 127);
  // 2^-e exactly (normal for e <= 126, the subnormal 2^-127 for e = 127)
  const float inv = e <= 126 ? __uint_as_float((uint32_t)(127 - e) << 23) : __uint_as_float(0x00400000u);
  const uint8_t c = (uint8_t)__nv_cvt_float_to_fp8(v * inv, __NV_SATFINITE, __NV_E4M3);
  return c == 0x80 ? 0 : c;  // a zero is stored as +0
}

// Barrier of one warpgroup (ids 1 and 2 as immediates, so that the kernel reserves three
// hardware barriers rather than all sixteen), optionally AND-reducing a predicate.
DSA_DEV void wg_barrier(int wg) {
  if (wg == 0)
    asm volatile("bar.sync 1, 128;" ::: "memory");
  else
    asm volatile("bar.sync 2, 128;" ::: "memory");
}
DSA_DEV bool wg_barrier_and(int wg, bool v) {
  uint32_t r;
  if (wg == 0)
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 128, p;\n"
                 " selp.u32 %0, 1, 0, q;\n}\n" : "=r"(r) : "r"((uint32_t)v) : "memory");
  else
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 2, 128, p;\n"
                 " selp.u32 %0, 1, 0, q;\n}\n" : "=r"(r) : "r"((uint32_t)v) : "memory");
  return r != 0;
}

// Split cluster barrier, arrive side without release semantics (what it orders is published by
// its own fence: the barriers' initialisation, or remote stores counted on mbarriers).
DSA_DEV void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }

// The same shared::cta address in CTA `rank` of the cluster (shared::cluster window).
DSA_DEV uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__global__ void __launch_bounds__(kThreads)
    prolog_kernel(const __grid_constant__ CUtensorMap tm_wq, const __grid_constant__ CUtensorMap tm_wk,
                  const __grid_constant__ CUtensorMap tm_ww, const __grid_constant__ CUtensorMap tm_xq,
                  const __grid_constant__ CUtensorMap tm_x, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from smem_raw by pointer arithmetic so that the compiler
  // keeps every access below in the shared state space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* recv = reinterpret_cast<float*>(smem + kStages * p.stage_max);  // [2][nrw][P][128]
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kStages * p.stage_max + p.recv_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = tid >> 7, f = tid & 127, qw = warp & 3;

  // ---- role, tile and slice of this CTA (a cluster: S consecutive CTAs of one role).  The K
  // and W tiles come first in the grid: their slices are the longest and they start first.
  int rb = blockIdx.x, role, P, nunits, nchunk, ntok;
  if (rb < 2 * p.ctas_k) {
    role = rb < p.ctas_k ? 1 : 2;
    if (role == 2) rb -= p.ctas_k;
    P = p.P_kw; nunits = p.units_k; nchunk = p.chunks_kw; ntok = p.ntok_kw;
  } else {
    rb -= 2 * p.ctas_k;
    role = 0; P = p.P_q; nunits = p.units_q; nchunk = p.chunks_q; ntok = p.ntok_q;
  }
  const int lg = 31 - __clz(ntok);         // ntok = 2^lg
  const int S = p.S, rank = rb % S;        // rank = %cluster_ctarank
  const int unit0 = (rb / S) * (S / P);    // first tile of the cluster
  const int unit = unit0 + rank / P, split = rank % P;
  const bool active = unit < nunits;       // the last cluster of a role may end in padding
  // a Q tile is (head, token tile); a K or W tile is a token tile
  const int head = role == 0 ? unit & 63 : 0;
  const int tok0 = (role == 0 ? unit >> 6 : unit) * ntok;
  // this slice's input chunks: an even share of the tile's, at least one
  const int c0 = (int)((long long)split * nchunk / P);
  const int n = (int)((long long)(split + 1) * nchunk / P) - c0;
  const int tmem_cols = ntok <= 32 ? 32 : (ntok <= 64 ? 64 : 128);
  const int stage_bytes = kATileBytes + ntok * 128;
  const CUtensorMap* tmA = role == 0 ? &tm_wq : (role == 1 ? &tm_wk : &tm_ww);
  const CUtensorMap* tmB = role == 0 ? &tm_xq : &tm_x;
  const uint32_t a_bytes = (role == 2 ? (uint32_t)p.H_I : 128u) * 128u;
  // rows of the cluster (its tiles' tokens, tile-major); warpgroup gw finishes gw, gw + 2S, ...
  const int R = (S / P) * ntok, gw = rank * 2 + wg, rstep = 2 * S;
  const int nrw = (ntok + 2 * P - 1) / (2 * P);  // rows per warpgroup at most

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->done, 1);
    ctl->abort = 0;
    for (int w = 0; w < 2; ++w) {
      // the bytes warpgroup w receives: P partial rows of 128 fp32 for each of its rows
      int rows = 0;
      for (int r = rank * 2 + w; r < R; r += rstep) rows += unit0 + (r >> lg) < nunits;
      mbar_init(&ctl->recv[w], 1);
      mbar_arrive_expect_tx(&ctl->recv[w], (uint32_t)(rows * P * 128 * 4));
    }
    fence_barrier_init();
  }
  if (warp == 1 && active) {
    tmem_alloc(&ctl->tmem_base, (uint32_t)tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive_relaxed();  // barriers initialised and armed (waited on before the first remote store)
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  // K tiles: the key-cache row of each row this CTA's warpgroups finish, resolved while the
  // projection streams (dependent loads: sequence of the token, its position, the page table)
  if (role == 1 && tid >= 64) {
    for (int e = tid - 64; e < 2 * kMaxOwnRows; e += kThreads - 64) {
      const int w2 = e / kMaxOwnRows, i = e - w2 * kMaxOwnRows;
      const int r = rank * 2 + w2 + i * rstep;
      if (r >= R) continue;  // (never read)
      const int u = unit0 + (r >> lg), t = u * ntok + (r & (ntok - 1));
      long long row = -1;
      if (u < nunits && t < p.n_q) {
        const int b = find_seq(p.q_start, p.B, t);
        const int pos = p.seq_lens[b] - (p.q_start[b + 1] - p.q_start[b]) + (t - p.q_start[b]);
        const int pg = (pos >= 0 && (pos >> 6) < p.max_pages) ? p.page_table[(size_t)b * p.max_pages + (pos >> 6)] : -1;
        if (pg >= 0 && pg < p.num_pages) row = (long long)pg * 64 + (pos & 63);
        else report(p.status, kStatusDeviceCheck);
      }
      ctl->krow[w2][i] = row;
    }
  }
  // K tiles: LayerNorm parameters of this thread's feature (a load only stalls where it is used)
  float ln_g = 0.f, ln_b = 0.f;
  if (role == 1) {
    ln_g = p.ln_gamma[f];
    ln_b = p.ln_beta[f];
  }

  // ---- the slice's projection: TMA ring (warp 0) -> tcgen05.mma into tensor memory (warp 1)
  bool stream_ok = true;
  if (active) {
    if (warp == 0 && lane == 0) {
      prefetch_tmap(tmA);
      prefetch_tmap(tmB);
      for (int i = 0; i < n; ++i) {
        const int s = i % kStages;
        if (i >= kStages && !mbar_wait(&ctl->empty[s], ((uint32_t)(i / kStages) & 1u) ^ 1u, abort, p.status))
          break;
        uint8_t* st = smem + (size_t)s * stage_bytes;
        mbar_arrive_expect_tx(&ctl->full[s], a_bytes + (uint32_t)ntok * 128u);
        tma_load_2d(st, tmA, &ctl->full[s], (c0 + i) * kChunk, head * 128);
        tma_load_2d(st + kATileBytes, tmB, &ctl->full[s], (c0 + i) * kChunk, tok0);
      }
      // never leave with copies in flight
      for (int i = max(0, n - kStages); i < n; ++i)
        mbar_wait(&ctl->full[i % kStages], (uint32_t)(i / kStages) & 1u, abort, p.status);
    } else if (warp == 1 && lane == 0) {
      const uint32_t idesc = idesc_bf16(128, ntok);
      const uint32_t base = smem_u32(smem);
      for (int i = 0; i < n; ++i) {
        const int s = i % kStages;
        if (!mbar_wait(&ctl->full[s], (uint32_t)(i / kStages) & 1u, abort, p.status)) break;
        tc_fence_after();
        const uint32_t st = base + (uint32_t)(s * stage_bytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 16 elements (32 bytes) of the 128-byte row per MMA
          mma_f16_ss(tmem, sdesc_sw128(st + kk * 32u, 16, 1024),
                     sdesc_sw128(st + kATileBytes + kk * 32u, 16, 1024), idesc,
                     (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&ctl->empty[s]);
      }
      mma_commit(&ctl->done);
    }
    // one thread waits for the accumulator; the others sleep in the block barrier below
    if (tid == 64) stream_ok = mbar_wait(&ctl->done, 0, abort, p.status);
  }
  // block-uniform: the accumulator is complete and nothing timed out
  const bool run = __syncthreads_and(stream_ok && *abort == 0) != 0;
  tc_fence_after();

  // ---- push each row of the partial tile to the warpgroup that finishes it
  cluster_wait();
  if (active && run) {
    const uint32_t lanes = tmem + ((uint32_t)(qw * 32) << 16);
    const uint32_t recv_a = smem_u32(recv), bar_a = smem_u32(&ctl->recv[0]);
    const int row0 = (rank / P) * ntok;  // this tile's first row in the cluster
    for (int j0 = wg * kGroupTok; j0 < ntok; j0 += kTokBlock) {
      uint32_t r[kGroupTok];
      tmem_ld_x8(lanes + (uint32_t)j0, r);
      // row row0 + j0 + i goes to warpgroup go of the cluster, into its row slot `slot`
      int go = (row0 + j0) % rstep, slot = (row0 + j0) / rstep;
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < kGroupTok; ++i) {
        const uint32_t owner = (uint32_t)(go >> 1), wo = (uint32_t)(go & 1);
        const uint32_t off = (uint32_t)(((((int)wo * nrw + slot) * P + split) * 128 + f) * 4);
        st_async_b32(map_rank(recv_a + off, owner), r[i], map_rank(bar_a + wo * 8u, owner));
        if (++go == rstep) {
          go = 0;
          ++slot;
        }
      }
    }
  }
  cluster_arrive_relaxed();  // this CTA's remote stores are issued

  // ---- this warpgroup's rows, kRowBatch at a time (every branch below is warpgroup-uniform)
  bool recv_ok = false;
  if (gw < R) {  // one thread of the warpgroup waits; the others sleep in its barrier
    bool ok = true;
    if (f == 0) ok = mbar_wait<true>(&ctl->recv[wg], 0, abort, p.status);
    recv_ok = wg_barrier_and(wg, ok);
  }
  const float* mine = recv + (size_t)wg * nrw * P * 128 + f;
  for (int r0 = gw, it = 0; r0 < R; r0 += rstep * kRowBatch, ++it) {
    float v[kRowBatch];
    bool rv[kRowBatch];
    int rt[kRowBatch], rh[kRowBatch];
#pragma unroll
    for (int b = 0; b < kRowBatch; ++b) {
      const int r = r0 + b * rstep, ul = r >> lg, j = r & (ntok - 1), u = unit0 + ul;
      rv[b] = recv_ok && r < R && u < nunits;
      rt[b] = (role == 0 ? u >> 6 : u) * ntok + j;  // token
      rh[b] = u & 63;                                // head (Q)
      // the sum of the slices' partial rows, in slice order
      float acc = 0.f;
      if (rv[b]) {
        const float* x = mine + (size_t)(it * kRowBatch + b) * P * 128;
        int sl = 0;
        for (; sl + 4 <= P; sl += 4) {  // four loads in flight, added in slice order
          const float a0 = x[sl * 128], a1 = x[(sl + 1) * 128], a2 = x[(sl + 2) * 128], a3 = x[(sl + 3) * 128];
          acc = (((acc + a0) + a1) + a2) + a3;
        }
        for (; sl < P; ++sl) acc += x[sl * 128];
      }
      v[b] = acc;
    }
    if (role == 1) {  // LayerNorm statistics of each row over its 128 features (rows of the
                      // batch that do not exist are skipped: rv is warpgroup-uniform)
#pragma unroll
      for (int b = 0; b < kRowBatch; ++b) {
        if (!rv[b]) continue;
        const float s = warp_sum(v[b]);
        if (lane == 0) ctl->red[0][warp][b] = s;
      }
      wg_barrier(wg);
#pragma unroll
      for (int b = 0; b < kRowBatch; ++b) {
        if (!rv[b]) continue;
        const float mean = (ctl->red[0][wg * 4][b] + ctl->red[0][wg * 4 + 1][b] + ctl->red[0][wg * 4 + 2][b] +
                            ctl->red[0][wg * 4 + 3][b]) * (1.f / 128.f);
        v[b] -= mean;
        const float s = warp_sum(v[b] * v[b]);
        if (lane == 0) ctl->red[1][warp][b] = s;
      }
      wg_barrier(wg);
#pragma unroll
      for (int b = 0; b < kRowBatch; ++b) {
        if (!rv[b]) continue;
        const float var = (ctl->red[1][wg * 4][b] + ctl->red[1][wg * 4 + 1][b] + ctl->red[1][wg * 4 + 2][b] +
                           ctl->red[1][wg * 4 + 3][b]) * (1.f / 128.f);
        v[b] = v[b] * __frsqrt_rn(var + p.ln_eps) * ln_g + ln_b;
      }
      // (red[0] is rewritten only after every thread has passed the second barrier, red[1]
      // only after the next batch's first one)
    }
#pragma unroll
    for (int b = 0; b < kRowBatch; ++b) {
      const int t = rt[b];
      if (!rv[b] || t >= p.n_q) continue;
      if (role == 2) {
        if (f < p.H_I) p.w_out[(size_t)t * p.H_I + f] = v[b] * p.w_scale;
        continue;
      }
      // destination row: q[t][head][:] or the key-cache row of the token's position
      const long long row = role == 0 ? (long long)t * p.H_I + rh[b] : ctl->krow[wg][it * kRowBatch + b];
      uint8_t* dst = role == 0 ? p.q_out : p.k_pool;
      uint8_t* sfdst = role == 0 ? p.q_sf : p.k_sf;
      if (p.mx) {
        uint8_t sf;
        const uint8_t c = mx_quant_lane(v[b], &sf);
        if (row >= 0) {
          dst[(size_t)row * 128 + f] = c;
          if (lane == 0) sfdst[(size_t)row * 4 + qw] = sf;
        }
      } else if (row >= 0) {
        reinterpret_cast<__nv_bfloat16*>(dst)[(size_t)row * 128 + f] = __float2bfloat16_rn(v[b]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1 && active) {
    __syncwarp();
    tmem_dealloc(tmem, (uint32_t)tmem_cols);
  }
  cluster_wait();  // every CTA of the cluster has issued its stores into this one
}

}  // namespace prolog

namespace prolog {

struct Plan {
  int ntok_q, ntok_kw, tiles_q, tiles_kw, chunks_q, chunks_kw;
  int S, P_q, P_kw, units_q, units_k, ctas_q, ctas_k, stage_max, recv_bytes, smem;
};

// Clusters of S CTAs with `smem` bytes each that the device keeps resident at once (0: none).
static int active_clusters(const DeviceInfo& dev, int S, int smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, int> memo;
  const auto key = std::make_tuple(dev.device, S, smem);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find(key);
    if (it != memo.end()) return it->second;
  }
  cudaLaunchConfig_t q = {};
  q.gridDim = dim3((unsigned)S);
  q.blockDim = dim3(kThreads);
  q.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)S;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  q.attrs = at;
  q.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, prolog_kernel, &q) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  memo[key] = n;
  return n;
}

// Tile sizes, slices per tile and cluster size.  Candidates: K / W tiles of 16 tokens or of the
// Q tiles' width; every cluster size S the device co-schedules, with slice counts P_q, P_kw that
// divide it (S their least common multiple, at most one slice per input chunk).  The estimate:
// each wave lasts as long as its longest slice streams at a CTA's share of the HBM (about
// 30 GB/s with two CTAs per SM) or as the wave's bytes take at the HBM rate, whichever is
// longer; the exchange of partial rows and the epilogue add a term per batch of rows.
static bool make_plan(const dsa_prolog_args& a, const DeviceInfo& dev, Plan& best, std::string& err) {
  const int chunks_q = (a.d_q + kChunk - 1) / kChunk;
  const int chunks_kw = (a.d_model + kChunk - 1) / kChunk;
  int ntok_q = 16;  // a power of two: 16 ... 128
  while (ntok_q < a.n_q && ntok_q < 128) ntok_q *= 2;
  const int tiles_q = (a.n_q + ntok_q - 1) / ntok_q;
  const int units_q = a.H_I * tiles_q;
  const double r_cta = 30e9, hbm = 6.4e12, t_batch = 1.6e-6, t_exchange = 0.9e-6;
  double best_est = 1e300;
  best = Plan{};
  int kw_opts[2] = {a.n_q <= 128 ? 16 : 128, ntok_q};
  for (int o = 0; o < 2; ++o) {
    const int ntok_kw = kw_opts[o];
    if (o == 1 && ntok_kw == kw_opts[0]) break;
    const int tiles_kw = (a.n_q + ntok_kw - 1) / ntok_kw;
    const int stage_max = kATileBytes + std::max(ntok_q, ntok_kw) * 128;
    for (int S = 1; S <= kMaxCluster; ++S) {
      for (int pq = 1; pq <= S; ++pq) {
        if (S % pq || pq > chunks_q) continue;
        for (int pk = 1; pk <= S; ++pk) {
          if (S % pk || pk > chunks_kw) continue;
          // S must be the least common multiple of the two slice counts
          int l = pq;
          while (l % pk) l += pq;
          if (l != S) continue;
          const long long ctas_q = (long long)((units_q + S / pq - 1) / (S / pq)) * S;
          const long long ctas_k = (long long)((tiles_kw + S / pk - 1) / (S / pk)) * S;
          const long long clusters = (ctas_q + 2 * ctas_k) / S;
          if (ctas_q + 2 * ctas_k > 0x7fffffffLL) continue;
          const int nrq = (ntok_q + 2 * pq - 1) / (2 * pq), nrk = (ntok_kw + 2 * pk - 1) / (2 * pk);
          const int recv_bytes = std::max(2 * nrq * pq, 2 * nrk * pk) * 128 * 4;
          const int smem = kStages * stage_max + recv_bytes + (int)sizeof(Ctl) + 1024;
          if (smem > dev.smem_optin) continue;
          // Clusters per wave.  The occupancy query counts one CTA per SM for a cluster; up to
          // 8 CTAs per cluster the hardware was measured to co-schedule every CTA that fits an
          // SM (e.g. 36 clusters of 8 at two CTAs per SM), beyond 8 about the query's count per
          // CTA slot of an SM.
          const int q_act = active_clusters(dev, S, smem);
          if (q_act <= 0) continue;
          const int per_sm = std::max(1, std::min(2048 / kThreads, dev.smem_per_sm / (smem + 1024)));
          const long long nact = S <= 8 ? std::max(1LL, (long long)dev.sm_count * per_sm / S)
                                        : (long long)q_act * per_sm;
          const double bq = (double)((chunks_q + pq - 1) / pq) * (kATileBytes + ntok_q * 128);
          const double bk = (double)((chunks_kw + pk - 1) / pk) * (kATileBytes + ntok_kw * 128);
          const double bytes = (double)ctas_q * bq + 2.0 * ctas_k * bk;
          const long long waves = (clusters + nact - 1) / nact;
          const double t_stream = waves * std::max(std::max(bq, bk) / r_cta, bytes / waves / hbm);
          const int rows = std::max(nrq, nrk);
          const double t_tail = t_exchange + ((rows + kRowBatch - 1) / kRowBatch) * t_batch;
          const double est = t_stream + waves * t_tail;
          if (est < best_est * 0.995) {
            best_est = est;
            best = Plan{ntok_q, ntok_kw, tiles_q, tiles_kw, chunks_q, chunks_kw, S, pq, pk,
                        units_q, tiles_kw, (int)ctas_q, (int)ctas_k, stage_max, recv_bytes, smem};
          }
        }
      }
    }
  }
  if (!best.S) {
    err = "indexer_prolog: no cluster shape fits the device";
    return false;
  }
  return true;
}

}  // namespace prolog

size_t prolog_workspace_bytes(const dsa_prolog_args&) { return 0; }

dsa_status launch_prolog(const dsa_prolog_args& a, cudaStream_t stream, std::string& err) {
  using namespace prolog;
  if (a.n_q == 0) return DSA_OK;
  DeviceInfo dev;
  if (!device_info(dev, err)) return DSA_ERR_CUDA;
  cudaError_t e = cudaFuncSetAttribute(prolog_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.smem_optin);
  if (e != cudaSuccess) return cuda_fail(e, "indexer_prolog: set shared memory size", err);
  e = cudaFuncSetAttribute(prolog_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return cuda_fail(e, "indexer_prolog: allow cluster > 8", err);
  // all of the unified L1 / shared memory as shared memory, so that the occupancy query counts
  // two CTAs per SM where their shared memory fits
  e = cudaFuncSetAttribute(prolog_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return cuda_fail(e, "indexer_prolog: shared memory carveout", err);
  Plan pl;
  if (!make_plan(a, dev, pl, err)) return DSA_ERR_UNSUPPORTED;
  CUtensorMap tm_wq, tm_wk, tm_ww, tm_xq, tm_x;
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!encode_tmap_2d(&tm_wq, bf, a.w_q, a.d_q, (uint64_t)a.H_I * a.d_I, (uint64_t)a.d_q * 2, kChunk, 128, sw, err) ||
      !encode_tmap_2d(&tm_wk, bf, a.w_k, a.d_model, a.d_I, (uint64_t)a.d_model * 2, kChunk, 128, sw, err) ||
      !encode_tmap_2d(&tm_ww, bf, a.w_w, a.d_model, a.H_I, (uint64_t)a.d_model * 2, kChunk, a.H_I, sw, err) ||
      !encode_tmap_2d(&tm_xq, bf, a.xq, a.d_q, a.n_q, (uint64_t)a.d_q * 2, kChunk, pl.ntok_q, sw, err) ||
      !encode_tmap_2d(&tm_x, bf, a.x, a.d_model, a.n_q, (uint64_t)a.d_model * 2, kChunk, pl.ntok_kw, sw, err))
    return DSA_ERR_CUDA;

  Params p{};
  p.n_q = a.n_q;
  p.B = a.B;
  p.H_I = a.H_I;
  p.mx = a.dtype == DSA_MXFP8_E4M3;
  p.ntok_q = pl.ntok_q;
  p.ntok_kw = pl.ntok_kw;
  p.tiles_q = pl.tiles_q;
  p.tiles_kw = pl.tiles_kw;
  p.stage_max = pl.stage_max;
  p.S = pl.S;
  p.P_q = pl.P_q;
  p.P_kw = pl.P_kw;
  p.units_q = pl.units_q;
  p.units_k = pl.units_k;
  p.ctas_q = pl.ctas_q;
  p.ctas_k = pl.ctas_k;
  p.chunks_q = pl.chunks_q;
  p.chunks_kw = pl.chunks_kw;
  p.recv_bytes = pl.recv_bytes;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.ln_eps = a.ln_eps;
  p.w_scale = a.w_scale;
  p.ln_gamma = a.ln_gamma;
  p.ln_beta = a.ln_beta;
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.q_start = a.q_start;
  p.q_out = reinterpret_cast<uint8_t*>(a.q_out);
  p.q_sf = a.q_sf;
  p.w_out = a.w_out;
  p.k_pool = reinterpret_cast<uint8_t*>(a.k_pool);
  p.k_sf = a.k_sf;
  p.status = a.status;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pl.ctas_q + 2 * pl.ctas_k));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)pl.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, prolog_kernel, tm_wq, tm_wk, tm_ww, tm_xq, tm_x, p);
  if (e != cudaSuccess) return cuda_fail(e, "indexer_prolog: launch", err);
  return DSA_OK;
}

}  // namespace dsa
