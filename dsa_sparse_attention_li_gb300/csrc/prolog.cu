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
// TMA into a 4-stage ring, warp 1 issues tcgen05.mma (bf16, fp32 accumulator in tensor memory);
// both warpgroups then share the epilogue, each taking half of every block of 16 tokens.
// With one slice per tile the CTA applies the epilogue straight from tensor memory; otherwise each
// slice stores its partial tile in the workspace and the last slice to arrive (arrival counter)
// adds the partials in slice order -- deterministic -- and applies the epilogue:
//   Q tiles (one per index head: 128 features = d_I): one warp holds one 32-feature group, so
//     the MX shared exponent is a warp max; e4m3 rounding to nearest even with saturation;
//   K tiles: LayerNorm over the 128 features (block reduction), quantisation, and the store of
//     the key row at the token's physical cache row (page table);
//   W tiles: the head weights (H_I = 64 rows of the tile).
#include <cuda_fp8.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace prolog {

constexpr int kThreads = 256;           // two warpgroups: each owns one lane quadrant per warp
constexpr int kGroupTok = 8;            // tokens of an epilogue block per warpgroup
constexpr int kChunk = 64;                // input elements per ring step (a 128-byte bf16 row)
constexpr int kStages = 4;
constexpr int kATileBytes = 128 * 128;    // 128 weight rows x 128 B
constexpr int kTokBlock = 16;             // tokens per epilogue pass (8 per warpgroup)

struct Params {
  int n_q, B, H_I, mx;
  int ntok_q, ntok_kw;          // tokens per tile (MMA N) of the Q tiles and of the K / W tiles
  int tiles_q, tiles_kw;        // token tiles of each
  int stage_max;                // ring stage bytes of the widest role
  int units_q, units_k;         // Q units = H_I * tiles_q; K units = W units = tiles_kw
  int splits_q, splits_kw;      // input slices per tile
  int chunks_q, chunks_kw;      // input chunks of the Q and of the K / W projections
  int per_q, per_kw;            // chunks per slice
  int ctas_q, ctas_k;           // grid: [Q CTAs][K CTAs][W CTAs]
  size_t off_q, off_k, off_w;  // float offsets of each role's partial tiles in the workspace
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
  float* ws;                    // partial tiles [role offset + slot][ntok][128]
  unsigned* counters;           // [units_q + 2 * units_k], zero between launches
  int* status;
};

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
  int last;
  float red[2][kThreads / 32][kGroupTok];  // LayerNorm sums: [sum | squares][warp][token]
  long long krow[128];  // K tiles: key-cache row of each token of the tile (-1: none / invalid)
};

struct Plan {
  int ntok_q, ntok_kw, tiles_q, tiles_kw, chunks_q, chunks_kw, splits_q, splits_kw, per_q, per_kw;
  int units_q, units_k, ctas_q, ctas_k, stage_max, smem;
  size_t off_q, off_k, off_w, part_floats, ws_bytes;
};

static Plan make_plan(const dsa_prolog_args& a, int sm_count) {
  Plan pl{};
  pl.ntok_q = a.n_q <= 128 ? std::max(16, (a.n_q + 15) / 16 * 16) : 128;
  // the K / W tiles end in a one-CTA reduction and epilogue: for a decode batch, tiles of 16
  // tokens spread them over more CTAs
  pl.ntok_kw = a.n_q <= 128 ? 16 : 128;
  pl.tiles_q = (a.n_q + pl.ntok_q - 1) / pl.ntok_q;
  pl.tiles_kw = (a.n_q + pl.ntok_kw - 1) / pl.ntok_kw;
  pl.chunks_q = (a.d_q + kChunk - 1) / kChunk;
  pl.chunks_kw = (a.d_model + kChunk - 1) / kChunk;
  pl.units_q = a.H_I * pl.tiles_q;
  pl.units_k = pl.tiles_kw;
  // about two CTAs per SM over the whole grid; the K / W tiles get slices of the Q tiles' length
  const int target = 2 * std::max(1, sm_count);
  pl.splits_q = std::max(1, std::min(pl.chunks_q, target / std::max(1, pl.units_q)));
  pl.per_q = (pl.chunks_q + pl.splits_q - 1) / pl.splits_q;
  pl.splits_q = (pl.chunks_q + pl.per_q - 1) / pl.per_q;
  pl.ctas_q = pl.units_q * pl.splits_q;
  // K / W slices: at most 16 to add, and the whole grid in one wave when it fits
  const int room = std::max(2 * pl.units_k, target - pl.ctas_q);
  const int want_kw = std::min(16, std::max(1, room / (2 * pl.units_k)));
  pl.per_kw = std::max(pl.per_q, (pl.chunks_kw + want_kw - 1) / want_kw);
  pl.splits_kw = (pl.chunks_kw + pl.per_kw - 1) / pl.per_kw;
  pl.ctas_k = pl.units_k * pl.splits_kw;
  size_t next = 0;  // floats
  pl.off_q = next;
  if (pl.splits_q > 1) next += (size_t)pl.ctas_q * pl.ntok_q * 128;
  pl.off_k = next;
  if (pl.splits_kw > 1) next += (size_t)pl.ctas_k * pl.ntok_kw * 128;
  pl.off_w = next;
  if (pl.splits_kw > 1) next += (size_t)pl.ctas_k * pl.ntok_kw * 128;
  pl.part_floats = next;
  const size_t part = next * sizeof(float);
  const size_t counters = (size_t)(pl.units_q + 2 * pl.units_k) * sizeof(unsigned);
  pl.ws_bytes = (part + 255) / 256 * 256 + (counters + 255) / 256 * 256;
  pl.stage_max = kATileBytes + std::max(pl.ntok_q, pl.ntok_kw) * 128;
  pl.smem = kStages * pl.stage_max + (int)sizeof(Ctl) + 1024;
  return pl;
}

DSA_DEV int find_seq(const int* q_start, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {  // largest b with q_start[b] <= t
    const int mid = (lo + hi + 1) >> 1;
    if (q_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Warp-wide maximum of non-negative floats (their bit patterns order like the values).
DSA_DEV float warp_max_nonneg(float a) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(a)));
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

__global__ void __launch_bounds__(kThreads)
    prolog_kernel(const __grid_constant__ CUtensorMap tm_wq, const __grid_constant__ CUtensorMap tm_wk,
                  const __grid_constant__ CUtensorMap tm_ww, const __grid_constant__ CUtensorMap tm_xq,
                  const __grid_constant__ CUtensorMap tm_x, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kStages * p.stage_max);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- which tile, slice and role this CTA computes
  int bid = blockIdx.x, role, splits, per, nchunk, unit_global;
  size_t ws_off;
  if (bid < p.ctas_q) {
    role = 0; splits = p.splits_q; per = p.per_q; nchunk = p.chunks_q; ws_off = p.off_q;
  } else if (bid < p.ctas_q + p.ctas_k) {
    role = 1; bid -= p.ctas_q;
    splits = p.splits_kw; per = p.per_kw; nchunk = p.chunks_kw; ws_off = p.off_k;
  } else {
    role = 2; bid -= p.ctas_q + p.ctas_k;
    splits = p.splits_kw; per = p.per_kw; nchunk = p.chunks_kw; ws_off = p.off_w;
  }
  const int ntok = role == 0 ? p.ntok_q : p.ntok_kw;  // MMA N of this CTA's tile
  const int tmem_cols = ntok <= 32 ? 32 : (ntok <= 64 ? 64 : 128);
  const int stage_bytes = kATileBytes + ntok * 128;
  const int unit = bid / splits, split = bid % splits;
  unit_global = role == 0 ? unit : (role == 1 ? p.units_q + unit : p.units_q + p.units_k + unit);
  const int head = role == 0 ? unit / p.tiles_q : 0;
  const int tok0 = (role == 0 ? unit % p.tiles_q : unit) * ntok;
  const int c0 = split * per, c1 = min(nchunk, c0 + per), n = c1 - c0;
  const CUtensorMap* tmA = role == 0 ? &tm_wq : (role == 1 ? &tm_wk : &tm_ww);
  const CUtensorMap* tmB = role == 0 ? &tm_xq : &tm_x;
  const uint32_t a_bytes = (role == 2 ? (uint32_t)p.H_I : 128u) * 128u;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->done, 1);
    ctl->abort = 0;
    ctl->last = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, (uint32_t)tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  // K tiles: each token's key-cache row, resolved once per token while the projection streams
  // (dependent loads: sequence of the token, its position, the page table)
  if (role == 1 && tid >= 64 && tid - 64 < ntok) {
    for (int j = tid - 64; j < ntok; j += kThreads - 64) {
      const int t = tok0 + j;
      long long row = -1;
      if (t < p.n_q) {
        const int b = find_seq(p.q_start, p.B, t);
        const int pos = p.seq_lens[b] - (p.q_start[b + 1] - p.q_start[b]) + (t - p.q_start[b]);
        const int pg = (pos >= 0 && (pos >> 6) < p.max_pages) ? p.page_table[(size_t)b * p.max_pages + (pos >> 6)] : -1;
        if (pg >= 0 && pg < p.num_pages) row = (long long)pg * 64 + (pos & 63);
        else report(p.status, kStatusDeviceCheck);
      }
      ctl->krow[j] = row;
    }
  }

  // K tiles: LayerNorm parameters of this thread's feature, loaded while the projection streams
  float ln_g = 0.f, ln_b = 0.f;
  if (role == 1) {  // (a load only stalls where its value is used: in the epilogue)
    ln_g = p.ln_gamma[tid & 127];
    ln_b = p.ln_beta[tid & 127];
  }

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
  const bool done_ok = mbar_wait(&ctl->done, 0, abort, p.status);
  tc_fence_after();
  // block-uniform: every thread saw the accumulator complete and nothing timed out
  bool run_epilogue = __syncthreads_and(done_ok && *abort == 0) != 0;
  // epilogue: thread (warpgroup wg, feature f = lane quadrant of its warp) -- both warpgroups
  // read the same 128 TMEM lanes, each for its own half of every block of tokens
  const int wg = tid >> 7, f = tid & 127, qw = warp & 3;
  const uint32_t lanes = tmem + ((uint32_t)(qw * 32) << 16);
  const size_t tile_floats = (size_t)ntok * 128;
  if (splits > 1) {
    if (run_epilogue) {
      float* w = p.ws + ws_off + (size_t)(unit * splits + split) * tile_floats;
      for (int j0 = wg * kGroupTok; j0 < ntok; j0 += kTokBlock) {
        uint32_t r[kGroupTok];
        tmem_ld_x8(lanes + (uint32_t)j0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kGroupTok; ++i) w[(size_t)(j0 + i) * 128 + f] = __uint_as_float(r[i]);
      }
      __threadfence();
    }
    __syncthreads();
    if (tid == 0 && run_epilogue) {
      const unsigned prev = atomicAdd(&p.counters[unit_global], 1u);
      ctl->last = prev == (unsigned)(splits - 1);
      if (ctl->last) p.counters[unit_global] = 0u;  // ready for the next launch
    }
    __syncthreads();
    run_epilogue = run_epilogue && ctl->last;
    if (run_epilogue) __threadfence();  // the other slices' partials are visible
  }

  float* tile = reinterpret_cast<float*>(smem);  // [ntok][128] sums (the ring is idle now)
  if (run_epilogue && splits > 1) {
    // add the slices' partial tiles in slice order; float4 loads, 8 x 4 in flight per thread
    const float4* part = reinterpret_cast<const float4*>(p.ws + ws_off + (size_t)(unit * splits) * tile_floats);
    const int n4 = ntok * 32;  // float4 per tile: a multiple of 512 = 2 * kThreads
    for (int e0 = tid; e0 < n4; e0 += 2 * kThreads) {
      float4 acc[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      int sl = 0;
      for (; sl + 8 <= splits; sl += 8) {
        float4 x[8][2];
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
          for (int u = 0; u < 2; ++u) x[q][u] = __ldcg(part + (size_t)(sl + q) * n4 + e0 + u * kThreads);
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            acc[u].x += x[q][u].x; acc[u].y += x[q][u].y; acc[u].z += x[q][u].z; acc[u].w += x[q][u].w;
          }
      }
      for (; sl < splits; ++sl)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float4 x = __ldcg(part + (size_t)sl * n4 + e0 + u * kThreads);
          acc[u].x += x.x; acc[u].y += x.y; acc[u].z += x.z; acc[u].w += x.w;
        }
#pragma unroll
      for (int u = 0; u < 2; ++u) reinterpret_cast<float4*>(tile)[e0 + u * kThreads] = acc[u];
    }
    __syncthreads();
  }
  if (run_epilogue) {
    for (int j0 = wg * kGroupTok; j0 < ntok; j0 += kTokBlock) {  // this warpgroup's 8 tokens
      float v[kGroupTok];
      if (splits == 1) {
        uint32_t r[kGroupTok];
        tmem_ld_x8(lanes + (uint32_t)j0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kGroupTok; ++i) v[i] = __uint_as_float(r[i]);
      } else {
#pragma unroll
        for (int i = 0; i < kGroupTok; ++i) v[i] = tile[(j0 + i) * 128 + f];
      }
      if (role == 1) {  // LayerNorm statistics of the block's tokens over the 128 features
        const float* r0 = ctl->red[0][wg * 4];
        const float* r1 = ctl->red[1][wg * 4];
#pragma unroll
        for (int i = 0; i < kGroupTok; ++i) {
          const float s = warp_sum(v[i]);
          if (lane == 0) ctl->red[0][warp][i] = s;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kGroupTok; ++i) {
          const float mean = (r0[i] + r0[kGroupTok + i] + r0[2 * kGroupTok + i] + r0[3 * kGroupTok + i]) * (1.f / 128.f);
          v[i] -= mean;
          const float s = warp_sum(v[i] * v[i]);
          if (lane == 0) ctl->red[1][warp][i] = s;
        }
        __syncthreads();
        const float g = ln_g, b = ln_b;
#pragma unroll
        for (int i = 0; i < kGroupTok; ++i) {
          const float var = (r1[i] + r1[kGroupTok + i] + r1[2 * kGroupTok + i] + r1[3 * kGroupTok + i]) * (1.f / 128.f);
          v[i] = v[i] * __frsqrt_rn(var + p.ln_eps) * g + b;
        }
        __syncthreads();  // red[] is reused by the next block
      }
      // the block's tokens are independent: unrolled and branch-free so their reductions and
      // stores overlap (predicated on the token existing and having a destination row)
      if (role == 2) {
#pragma unroll
        for (int i = 0; i < kGroupTok; ++i) {
          const int t = tok0 + j0 + i;
          if (t < p.n_q && f < p.H_I) p.w_out[(size_t)t * p.H_I + f] = v[i] * p.w_scale;
        }
      } else {
        uint8_t* dst = role == 0 ? p.q_out : p.k_pool;
        uint8_t* sfdst = role == 0 ? p.q_sf : p.k_sf;
#pragma unroll
        for (int i = 0; i < kGroupTok; ++i) {
          const int t = tok0 + j0 + i;
          // destination row: q[t][head][:] or the key-cache row of the token's position
          const long long row = role == 0 ? (long long)t * p.H_I + head : ctl->krow[j0 + i];
          const bool store = t < p.n_q && row >= 0;
          if (p.mx) {
            uint8_t sf;
            const uint8_t c = mx_quant_lane(v[i], &sf);
            if (store) dst[(size_t)row * 128 + f] = c;
            if (store && lane == 0) sfdst[(size_t)row * 4 + qw] = sf;
          } else if (store) {
            reinterpret_cast<__nv_bfloat16*>(dst)[(size_t)row * 128 + f] = __float2bfloat16_rn(v[i]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, (uint32_t)tmem_cols);
  }
}

}  // namespace prolog

size_t prolog_workspace_bytes(const dsa_prolog_args& a) {
  DeviceInfo dev;
  std::string err;
  if (!device_info(dev, err)) return 0;
  return prolog::make_plan(a, dev.sm_count).ws_bytes;
}

dsa_status launch_prolog(const dsa_prolog_args& a, cudaStream_t stream, std::string& err) {
  using namespace prolog;
  if (a.n_q == 0) return DSA_OK;
  DeviceInfo dev;
  if (!device_info(dev, err)) return DSA_ERR_CUDA;
  const Plan pl = make_plan(a, dev.sm_count);
  if (a.workspace_bytes < pl.ws_bytes) {
    err = "indexer_prolog: workspace_bytes below dsa_prolog_workspace_bytes()";
    return DSA_ERR_INVALID_ARG;
  }
  if (pl.smem > dev.smem_optin) {
    err = "indexer_prolog: shared memory";
    return DSA_ERR_UNSUPPORTED;
  }
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
  p.units_q = pl.units_q;
  p.units_k = pl.units_k;
  p.splits_q = pl.splits_q;
  p.splits_kw = pl.splits_kw;
  p.chunks_q = pl.chunks_q;
  p.chunks_kw = pl.chunks_kw;
  p.per_q = pl.per_q;
  p.per_kw = pl.per_kw;
  p.ctas_q = pl.ctas_q;
  p.ctas_k = pl.ctas_k;
  p.off_q = pl.off_q;
  p.off_k = pl.off_k;
  p.off_w = pl.off_w;
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
  const size_t part = pl.part_floats * sizeof(float);
  p.ws = reinterpret_cast<float*>(a.workspace);
  p.counters = reinterpret_cast<unsigned*>(reinterpret_cast<uint8_t*>(a.workspace) + (part + 255) / 256 * 256);
  p.status = a.status;

  cudaError_t e = cudaFuncSetAttribute(prolog_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return cuda_fail(e, "indexer_prolog: set shared memory size", err);
  const unsigned grid = (unsigned)(pl.ctas_q + 2 * pl.ctas_k);
  prolog_kernel<<<grid, kThreads, pl.smem, stream>>>(tm_wq, tm_wk, tm_ww, tm_xq, tm_x, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "indexer_prolog: launch", err);
  return DSA_OK;
}

}  // namespace dsa
