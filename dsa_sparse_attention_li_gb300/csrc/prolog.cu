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

constexpr int kThreads = 128;
constexpr int kChunk = 64;                // input elements per ring step (a 128-byte bf16 row)
constexpr int kStages = 4;
constexpr int kATileBytes = 128 * 128;    // 128 weight rows x 128 B
constexpr int kTokBlock = 16;             // tokens per epilogue pass (one tcgen05.ld x16)

struct Params {
  int n_q, B, H_I, mx;
  int ntok, tok_tiles, tmem_cols;
  int units_q, units_k;         // Q units = H_I * tok_tiles; K units = W units = tok_tiles
  int splits_q, splits_kw;      // input slices per tile
  int chunks_q, chunks_kw;      // input chunks of the Q and of the K / W projections
  int per_q, per_kw;            // chunks per slice
  int ctas_q, ctas_k;           // grid: [Q CTAs][K CTAs][W CTAs]
  int slot_q, slot_k, slot_w;   // first workspace slot of each role
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
  float* ws;                    // partial tiles [slot][ntok][128]
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
  float red[2][kThreads / 32][kTokBlock];  // LayerNorm sums: [sum | squares][warp][token]
};

struct Plan {
  int ntok, tok_tiles, tmem_cols, chunks_q, chunks_kw, splits_q, splits_kw, per_q, per_kw;
  int units_q, units_k, ctas_q, ctas_k, slot_q, slot_k, slot_w, slots, smem;
  size_t ws_bytes;
};

static Plan make_plan(const dsa_prolog_args& a, int sm_count) {
  Plan pl{};
  pl.ntok = a.n_q <= 128 ? std::max(16, (a.n_q + 15) / 16 * 16) : 128;
  pl.tok_tiles = (a.n_q + pl.ntok - 1) / pl.ntok;
  pl.tmem_cols = 32;
  while (pl.tmem_cols < pl.ntok) pl.tmem_cols *= 2;
  pl.chunks_q = (a.d_q + kChunk - 1) / kChunk;
  pl.chunks_kw = (a.d_model + kChunk - 1) / kChunk;
  pl.units_q = a.H_I * pl.tok_tiles;
  pl.units_k = pl.tok_tiles;
  // about two CTAs per SM over the whole grid; the K / W tiles get slices of the Q tiles' length
  const int target = 2 * std::max(1, sm_count);
  pl.splits_q = std::max(1, std::min(pl.chunks_q, target / std::max(1, pl.units_q)));
  pl.per_q = (pl.chunks_q + pl.splits_q - 1) / pl.splits_q;
  pl.splits_q = (pl.chunks_q + pl.per_q - 1) / pl.per_q;
  pl.per_kw = std::max(pl.per_q, (pl.chunks_kw + 31) / 32);
  pl.splits_kw = (pl.chunks_kw + pl.per_kw - 1) / pl.per_kw;
  pl.ctas_q = pl.units_q * pl.splits_q;
  pl.ctas_k = pl.units_k * pl.splits_kw;
  int next = 0;
  pl.slot_q = next;
  if (pl.splits_q > 1) next += pl.ctas_q;
  pl.slot_k = next;
  if (pl.splits_kw > 1) next += pl.ctas_k;
  pl.slot_w = next;
  if (pl.splits_kw > 1) next += pl.ctas_k;
  pl.slots = next;
  const size_t part = (size_t)pl.slots * pl.ntok * 128 * sizeof(float);
  const size_t counters = (size_t)(pl.units_q + 2 * pl.units_k) * sizeof(unsigned);
  pl.ws_bytes = (part + 255) / 256 * 256 + (counters + 255) / 256 * 256;
  pl.smem = kStages * (kATileBytes + pl.ntok * 128) + (int)sizeof(Ctl) + 1024;
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
  const float amax = warp_max_nonneg(fabsf(v));
  int e = 0;
  if (amax > 0.f) {
    int ex;
    frexpf(amax, &ex);  // amax = m * 2^ex, m in [0.5, 1)
    e = min(127, max(-127, ex - 1 - 8));
  }
  *sf = (uint8_t)(e + 127);
  uint8_t c = (uint8_t)__nv_cvt_float_to_fp8(ldexpf(v, -e), __NV_SATFINITE, __NV_E4M3);
  return c == 0x80 ? 0 : c;  // a zero is stored as +0
}

__global__ void __launch_bounds__(kThreads)
    prolog_kernel(const __grid_constant__ CUtensorMap tm_wq, const __grid_constant__ CUtensorMap tm_wk,
                  const __grid_constant__ CUtensorMap tm_ww, const __grid_constant__ CUtensorMap tm_xq,
                  const __grid_constant__ CUtensorMap tm_x, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int stage_bytes = kATileBytes + p.ntok * 128;
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kStages * stage_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- which tile, slice and role this CTA computes
  int bid = blockIdx.x, role, splits, per, nchunk, slot_base, unit_global;
  if (bid < p.ctas_q) {
    role = 0; splits = p.splits_q; per = p.per_q; nchunk = p.chunks_q; slot_base = p.slot_q;
  } else if (bid < p.ctas_q + p.ctas_k) {
    role = 1; bid -= p.ctas_q;
    splits = p.splits_kw; per = p.per_kw; nchunk = p.chunks_kw; slot_base = p.slot_k;
  } else {
    role = 2; bid -= p.ctas_q + p.ctas_k;
    splits = p.splits_kw; per = p.per_kw; nchunk = p.chunks_kw; slot_base = p.slot_w;
  }
  const int unit = bid / splits, split = bid % splits;
  unit_global = role == 0 ? unit : (role == 1 ? p.units_q + unit : p.units_q + p.units_k + unit);
  const int head = role == 0 ? unit / p.tok_tiles : 0;
  const int tok0 = (role == 0 ? unit % p.tok_tiles : unit) * p.ntok;
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
    tmem_alloc(&ctl->tmem_base, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  if (warp == 0 && lane == 0) {
    prefetch_tmap(tmA);
    prefetch_tmap(tmB);
    for (int i = 0; i < n; ++i) {
      const int s = i % kStages;
      if (i >= kStages && !mbar_wait(&ctl->empty[s], ((uint32_t)(i / kStages) & 1u) ^ 1u, abort, p.status))
        break;
      uint8_t* st = smem + (size_t)s * stage_bytes;
      mbar_arrive_expect_tx(&ctl->full[s], a_bytes + (uint32_t)p.ntok * 128u);
      tma_load_2d(st, tmA, &ctl->full[s], (c0 + i) * kChunk, head * 128);
      tma_load_2d(st + kATileBytes, tmB, &ctl->full[s], (c0 + i) * kChunk, tok0);
    }
    // never leave with copies in flight
    for (int i = max(0, n - kStages); i < n; ++i)
      mbar_wait(&ctl->full[i % kStages], (uint32_t)(i / kStages) & 1u, abort, p.status);
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16(128, p.ntok);
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
  const uint32_t lanes = tmem + ((uint32_t)(warp * 32) << 16);
  const size_t tile_floats = (size_t)p.ntok * 128;
  if (splits > 1) {
    if (run_epilogue) {
      float* w = p.ws + (size_t)(slot_base + unit * splits + split) * tile_floats;
      for (int j0 = 0; j0 < p.ntok; j0 += kTokBlock) {
        uint32_t r[kTokBlock];
        tmem_ld_x16(lanes + (uint32_t)j0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kTokBlock; ++i) w[(size_t)(j0 + i) * 128 + tid] = __uint_as_float(r[i]);
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

  if (run_epilogue) {
    const float* part = p.ws + (size_t)(slot_base + unit * splits) * tile_floats;
    for (int j0 = 0; j0 < p.ntok; j0 += kTokBlock) {
      float v[kTokBlock];
      if (splits == 1) {
        uint32_t r[kTokBlock];
        tmem_ld_x16(lanes + (uint32_t)j0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kTokBlock; ++i) v[i] = __uint_as_float(r[i]);
      } else {
#pragma unroll
        for (int i = 0; i < kTokBlock; ++i) v[i] = 0.f;
        for (int s = 0; s < splits; ++s)  // fixed slice order
#pragma unroll
          for (int i = 0; i < kTokBlock; ++i)
            v[i] += __ldcg(part + (size_t)s * tile_floats + (size_t)(j0 + i) * 128 + tid);
      }
      if (role == 1) {  // LayerNorm statistics of the block's tokens over the 128 features
#pragma unroll
        for (int i = 0; i < kTokBlock; ++i) {
          const float s = warp_sum(v[i]);
          if (lane == 0) ctl->red[0][warp][i] = s;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kTokBlock; ++i) {
          const float mean = (ctl->red[0][0][i] + ctl->red[0][1][i] + ctl->red[0][2][i] + ctl->red[0][3][i]) * (1.f / 128.f);
          v[i] -= mean;
          const float s = warp_sum(v[i] * v[i]);
          if (lane == 0) ctl->red[1][warp][i] = s;
        }
        __syncthreads();
        const float g = p.ln_gamma[tid], b = p.ln_beta[tid];
#pragma unroll
        for (int i = 0; i < kTokBlock; ++i) {
          const float var = (ctl->red[1][0][i] + ctl->red[1][1][i] + ctl->red[1][2][i] + ctl->red[1][3][i]) * (1.f / 128.f);
          v[i] = v[i] * __frsqrt_rn(var + p.ln_eps) * g + b;
        }
        __syncthreads();  // red[] is reused by the next block
      }
#pragma unroll 1
      for (int i = 0; i < kTokBlock; ++i) {
        const int t = tok0 + j0 + i;  // uniform over the block
        if (t >= p.n_q) break;
        if (role == 2) {
          if (tid < p.H_I) p.w_out[(size_t)t * p.H_I + tid] = v[i] * p.w_scale;
          continue;
        }
        // destination of this token's row: q[t][head][:] or the key-cache row of its position
        size_t row;
        if (role == 0) {
          row = (size_t)t * p.H_I + head;
        } else {
          const int b = find_seq(p.q_start, p.B, t);
          const int pos = p.seq_lens[b] - (p.q_start[b + 1] - p.q_start[b]) + (t - p.q_start[b]);
          const int pg = (pos >= 0 && (pos >> 6) < p.max_pages) ? p.page_table[(size_t)b * p.max_pages + (pos >> 6)] : -1;
          if (pg < 0 || pg >= p.num_pages) {
            if (tid == 0) report(p.status, kStatusDeviceCheck);
            continue;
          }
          row = (size_t)pg * 64 + (pos & 63);
        }
        uint8_t* dst = role == 0 ? p.q_out : p.k_pool;
        if (p.mx) {
          uint8_t sf;
          const uint8_t c = mx_quant_lane(v[i], &sf);
          dst[row * 128 + tid] = c;
          if (lane == 0) (role == 0 ? p.q_sf : p.k_sf)[row * 4 + warp] = sf;
        } else {
          reinterpret_cast<__nv_bfloat16*>(dst)[row * 128 + tid] = __float2bfloat16_rn(v[i]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
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
      !encode_tmap_2d(&tm_xq, bf, a.xq, a.d_q, a.n_q, (uint64_t)a.d_q * 2, kChunk, pl.ntok, sw, err) ||
      !encode_tmap_2d(&tm_x, bf, a.x, a.d_model, a.n_q, (uint64_t)a.d_model * 2, kChunk, pl.ntok, sw, err))
    return DSA_ERR_CUDA;

  Params p{};
  p.n_q = a.n_q;
  p.B = a.B;
  p.H_I = a.H_I;
  p.mx = a.dtype == DSA_MXFP8_E4M3;
  p.ntok = pl.ntok;
  p.tok_tiles = pl.tok_tiles;
  p.tmem_cols = pl.tmem_cols;
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
  p.slot_q = pl.slot_q;
  p.slot_k = pl.slot_k;
  p.slot_w = pl.slot_w;
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
  const size_t part = (size_t)pl.slots * pl.ntok * 128 * sizeof(float);
  p.ws = reinterpret_cast<float*>(a.workspace);
  p.counters = reinterpret_cast<unsigned*>(reinterpret_cast<uint8_t*>(a.workspace) + (part + 255) / 256 * 256);
  p.status = a.status;

  cudaError_t e = cudaFuncSetAttribute(prolog_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
  if (e != cudaSuccess) return cuda_fail(e, "indexer_prolog: set shared memory size", err);
  const unsigned grid = (unsigned)(pl.ctas_q + 2 * pl.ctas_k);
  if (std::getenv("DSA_VERBOSE"))
    std::fprintf(stderr, "[dsa] prolog ntok=%d tiles=%d splits q=%d kw=%d (chunks %d/%d) grid=%u smem=%d ws=%zu\n",
                 pl.ntok, pl.tok_tiles, pl.splits_q, pl.splits_kw, pl.per_q, pl.per_kw, grid, pl.smem,
                 pl.ws_bytes);
  prolog_kernel<<<grid, kThreads, pl.smem, stream>>>(tm_wq, tm_wk, tm_ww, tm_xq, tm_x, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "indexer_prolog: launch", err);
  return DSA_OK;
}

}  // namespace dsa
