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
// Work decomposition.  A CTA serves one (query token, value half r, row split s):
//   - Q[t] (128 heads x 576, bf16) is staged once by TMA into a 128-byte-swizzled K-major tile;
//   - the split's selected positions are translated to physical rows (page table) in shared
//     memory, then each 32-row tile is gathered by TMA tile::gather4 (4 rows x 128 bytes per
//     instruction) into a 2-stage ring: the same swizzled tile serves as the K-major B operand of
//     Q.K^T (N = 32 rows, K = 576) and as the MN-major B operand of P.V (K = 32 rows, N = 256);
//   - S = Q.K^T goes to a double-buffered TMEM accumulator; one thread per head (TMEM lane) masks,
//     scales and exponentiates its row, writes P (bf16) back to TMEM and accumulates the row sum;
//     the reference maximum only moves when a tile's maximum exceeds it by more than 2^8, and only
//     then is the head's O row rescaled in TMEM;
//   - O (128 x 256 fp32 = half of TMEM) accumulates P.V_r across tiles.
// Each head's 128x512 fp32 O would fill all of TMEM, so the value columns are split over two
// CTAs (r = 0, 1) that recompute the same S.  With several row splits the partial (o, lse) are
// written to the caller's workspace and the last CTA of a (token, r) to finish merges them.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace sfa {

constexpr int kThreads = 256;
constexpr int kHeads = 128;        // MMA M (heads are padded to 128)
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kDvHalf = 256;
constexpr int kNT = 32;            // gathered rows per tile
constexpr int kStages = 2;
constexpr int kBoxes = kDqk / 64;  // 9 column boxes of 64 bf16 (128 B)
constexpr int kQBytes = kHeads * kDqk * 2;       // 147456
constexpr int kTileBytes = kNT * kDqk * 2;       // 36864
constexpr int kMaxRows = 2048;     // row slots per CTA
constexpr float kRescaleLog2 = 8.0f;
// TMEM columns
constexpr uint32_t kColS = 0;      // two 32-column S buffers
constexpr uint32_t kColP = 64;     // P: 32 bf16 per lane = 16 columns
constexpr uint32_t kColO = 256;    // O half: 256 columns
constexpr uint32_t kTmemCols = 512;

struct Params {
  int B, n_q, H, K, max_pages, num_pages;
  int splits;      // row splits per token
  int rows_per;    // row slots per split (multiple of kNT)
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
  const __nv_bfloat16* q;   // raw pointers for the CUDA-core variant
  const __nv_bfloat16* kv;
};

struct Layout {
  static constexpr int q = 0;
  static constexpr int stages = q + kQBytes;
  static constexpr int rows = stages + kStages * kTileBytes;
  static constexpr int ctl = rows + kMaxRows * 4;
  static constexpr int total = ctl + 512;
};

struct Ctl {
  uint64_t qbar;
  uint64_t full[kStages], empty[kStages];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, pv_done, drain;
  uint32_t tmem_base;
  int abort;
  int ntile;
  int last;  // this CTA merges the splits
  int nvalid;
};

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

__global__ void __launch_bounds__(kThreads, 1)
    sfa_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
               const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* q_s = smem + Layout::q;
  uint8_t* st_s = smem + Layout::stages;
  int* rows_s = reinterpret_cast<int*>(smem + Layout::rows);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + Layout::ctl);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x % p.splits;
  const int half = (blockIdx.x / p.splits) & 1;
  const int t = blockIdx.x / (2 * p.splits);
  if (t >= p.n_q) return;
  const int b = find_seq(p.q_start, p.B, t);
  const int L = p.seq_lens[b];
  const int slot0 = split * p.rows_per;
  const int nslot = max(0, min(p.rows_per, p.K - slot0));

  if (tid == 0) {
    mbar_init(&ctl->qbar, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->s_full[a], 1);
      mbar_init(&ctl->s_free[a], 128);
    }
    mbar_init(&ctl->p_full, 128);
    mbar_init(&ctl->pv_done, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    ctl->nvalid = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // logical position -> physical row of every slot of this split (-1: empty or invalid)
  int last_valid = -1;
  for (int i = tid; i < nslot; i += kThreads) {
    const int j = p.idx[(size_t)t * p.K + slot0 + i];
    int row = -1;
    if (j >= 0) {
      if (j < L) {
        const int pg = p.page_table[(size_t)b * p.max_pages + (j >> 6)];
        if (pg >= 0 && pg < p.num_pages)
          row = pg * 64 + (j & 63);
        else
          report(p.status, kStatusDeviceCheck);
      } else {
        report(p.status, kStatusDeviceCheck);
      }
    } else if (j < -1) {
      report(p.status, kStatusDeviceCheck);
    }
    rows_s[i] = row;
    if (row >= 0) last_valid = i;
  }
  // tiles needed: up to the last valid slot
  last_valid = __reduce_max_sync(0xffffffffu, last_valid + 1) - 1;
  if (lane == 0 && last_valid >= 0) atomicMax(&ctl->nvalid, last_valid + 1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int ntile = (ctl->nvalid + kNT - 1) / kNT;
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  float m_ref = -INFINITY, l_sum = 0.f;  // per-head state (threads 128..255)

  if (warp == 0 && lane == 0) {
    // ---------------- producer: Q once, then gathered tiles
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_kv);
    if (ntile > 0) {
      mbar_arrive_expect_tx(&ctl->qbar, kQBytes);
      for (int bx = 0; bx < kBoxes; ++bx)
        tma_load_2d(q_s + bx * (kHeads * 128), &tm_q, &ctl->qbar, bx * 64, t * p.H);
    }
    for (int i = 0; i < ntile; ++i) {
      const int s = i % kStages;
      if (i >= kStages &&
          !mbar_wait(&ctl->empty[s], ((uint32_t)(i / kStages) & 1u) ^ 1u, abort, p.status))
        break;
      mbar_arrive_expect_tx(&ctl->full[s], kTileBytes);
      uint8_t* dst = st_s + s * kTileBytes;
      for (int g = 0; g < kNT / 4; ++g) {
        int r[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int slot = i * kNT + 4 * g + k;
          const int row = slot < nslot ? rows_s[slot] : -1;
          r[k] = row >= 0 ? row : 0;  // empty slots read row 0; their weight is exactly 0
        }
#pragma unroll
        for (int bx = 0; bx < kBoxes; ++bx)
          tma_gather4(dst + bx * (kNT * 128) + g * 512, &tm_kv, &ctl->full[s], bx * 64, r[0], r[1],
                      r[2], r[3]);
      }
    }
    for (int i = max(0, ntile - kStages); i < ntile; ++i)
      mbar_wait(&ctl->full[i % kStages], (uint32_t)(i / kStages) & 1u, abort, p.status);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc_qk = idesc_bf16(128, kNT);
    constexpr uint32_t idesc_pv = idesc_bf16(128, kDvHalf, /*b_mn_major=*/true);
    const uint32_t q_addr = smem_u32(q_s), st_addr = smem_u32(st_s);
    bool ok = ntile == 0 || mbar_wait(&ctl->qbar, 0, abort, p.status);
    for (int i = 0; ok && i <= ntile; ++i) {
      if (i < ntile) {
        const int s = i % kStages, a = i & 1;
        if (!mbar_wait(&ctl->full[s], (uint32_t)(i / kStages) & 1u, abort, p.status)) break;
        if (i >= 2 && !mbar_wait(&ctl->s_free[a], ((uint32_t)(i >> 1) & 1u) ^ 1u, abort, p.status))
          break;
        tc_fence_after();
        const uint32_t d = tmem + kColS + (uint32_t)(a * kNT);
        const uint32_t sb = st_addr + (uint32_t)(s * kTileBytes);
#pragma unroll 4
        for (int kk = 0; kk < kDqk / 16; ++kk) {
          const uint32_t bx = (uint32_t)kk >> 2, off = ((uint32_t)kk & 3u) * 32u;
          const uint64_t ad = sdesc_sw128(q_addr + bx * (kHeads * 128) + off, 16, 1024);
          const uint64_t bd = sdesc_sw128(sb + bx * (kNT * 128) + off, 16, 1024);
          mma_f16_ss(d, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&ctl->s_full[a]);
      }
      if (i >= 1) {
        const int ip = i - 1, s = ip % kStages;
        if (!mbar_wait(&ctl->p_full, (uint32_t)ip & 1u, abort, p.status)) break;
        tc_fence_after();
        const uint32_t sb = st_addr + (uint32_t)(s * kTileBytes) + (uint32_t)(half * 4 * kNT * 128);
#pragma unroll
        for (int kk = 0; kk < kNT / 16; ++kk) {
          // B = V rows [16kk, 16kk+16) x this half's 256 value columns, MN-major:
          // 64-column blocks kNT*128 bytes apart (lbo), 8-row groups 1024 bytes apart (sbo)
          const uint64_t bd = sdesc_sw128(sb + (uint32_t)kk * 2048u, kNT * 128, 1024);
          mma_f16_ts(tmem + kColO, tmem + kColP + (uint32_t)kk * 8u, bd, idesc_pv,
                     (ip > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&ctl->pv_done);
        mma_commit(&ctl->empty[s]);
      }
    }
    mma_commit(&ctl->drain);
    mbar_wait(&ctl->drain, 0, abort, p.status);
  } else if (warp >= 4) {
    // ---------------- softmax: one thread per head row (TMEM lane)
    const int qd = warp - 4, h = qd * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(qd * 32) << 16);
    for (int i = 0; i < ntile; ++i) {
      const int a = i & 1;
      bool ok = mbar_wait(&ctl->s_full[a], (uint32_t)(i >> 1) & 1u, abort, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld_x32(lane_addr + kColS + (uint32_t)(a * kNT), sr);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&ctl->s_free[a]);
      float z[32];
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int slot = i * kNT + c;
        const bool valid = slot < nslot && rows_s[slot] >= 0;
        z[c] = valid ? __uint_as_float(sr[c]) * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, z[c]);
      }
      if (i >= 1) {
        ok = mbar_wait(&ctl->pv_done, (uint32_t)(i - 1) & 1u, abort, p.status);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
      }
      // lazy rescale: move the reference maximum only when it is exceeded by more than 2^8
      const bool need = mt > m_ref + kRescaleLog2;
      if (__any_sync(0xffffffffu, need && i >= 1 && l_sum > 0.f)) {
        const float alpha = (need && l_sum > 0.f) ? exp2f(m_ref - mt) : 1.f;
#pragma unroll 1
        for (int c = 0; c < kDvHalf / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(lane_addr + kColO + (uint32_t)(c * 32), o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st_x16(lane_addr + kColO + (uint32_t)(c * 32), o);
          tmem_st_x16(lane_addr + kColO + (uint32_t)(c * 32 + 16), o + 16);
        }
        tmem_st_wait();
        if (need) l_sum *= alpha;
      }
      if (need) m_ref = mt;
      uint32_t pk[16];
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float p0 = m_ref == -INFINITY ? 0.f : exp2f(z[2 * c] - m_ref);
        const float p1 = m_ref == -INFINITY ? 0.f : exp2f(z[2 * c + 1] - m_ref);
        pk[c] = pack_bf16(p0, p1);
        const __nv_bfloat162 r = *reinterpret_cast<__nv_bfloat162*>(&pk[c]);
        ls += __bfloat162float(r.x) + __bfloat162float(r.y);  // sum what P.V actually uses
      }
      l_sum += ls;
      tmem_st_x16(lane_addr + kColP, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ctl->p_full);
    }
    if (ntile > 0) {
      const bool ok = mbar_wait(&ctl->pv_done, (uint32_t)(ntile - 1) & 1u, abort, p.status);
      (void)__all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    // ---------------- epilogue
    const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
    const float lse2 = l_sum > 0.f ? m_ref + log2f(l_sum) : -INFINITY;
    if (p.splits == 1) {
      __nv_bfloat16* orow = p.out + ((size_t)t * p.H + h) * kDv + half * kDvHalf;
#pragma unroll 1
      for (int c = 0; c < kDvHalf / 32; ++c) {
        uint32_t o[32];
        if (ntile > 0) {
          tmem_ld_x32(lane_addr + kColO + (uint32_t)(c * 32), o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0u;
        }
        if (h < p.H) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            dst[v] = w;
          }
        }
      }
      if (half == 0 && h < p.H && p.lse) p.lse[(size_t)t * p.H + h] = lse2 * 0.69314718055994531f;
    } else {
      const size_t unit = ((size_t)t * 2 + half) * p.splits + split;
      float* po = p.ws_o + (unit * kHeads + h) * kDvHalf;
#pragma unroll 1
      for (int c = 0; c < kDvHalf / 32; ++c) {
        uint32_t o[32];
        if (ntile > 0) {
          tmem_ld_x32(lane_addr + kColO + (uint32_t)(c * 32), o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0u;
        }
        float4* dst = reinterpret_cast<float4*>(po + c * 32);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          __stcg(dst + v, make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                      __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv));
      }
      __stcg(p.ws_lse + unit * kHeads + h, lse2);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (p.splits == 1) return;

  // ---------------- last CTA of (token, half) merges the split partials
  if (tid == 0) {
    __threadfence();
    const int prev = atomicAdd(&p.ws_count[t * 2 + half], 1);
    ctl->last = prev == p.splits - 1;
    if (ctl->last) p.ws_count[t * 2 + half] = 0;  // ready for the next call
  }
  __syncthreads();
  if (!ctl->last) return;
  __threadfence();
  const size_t unit0 = ((size_t)t * 2 + half) * p.splits;
  // 256 threads: head h = tid / 2, value columns [128 * (tid & 1), +128)
  const int h = tid >> 1, c0 = (tid & 1) * 128;
  float M = -INFINITY;
  for (int s = 0; s < p.splits; ++s) M = fmaxf(M, __ldcg(p.ws_lse + (unit0 + s) * kHeads + h));
  float W = 0.f;
  float acc[128];
#pragma unroll
  for (int k = 0; k < 128; ++k) acc[k] = 0.f;
  for (int s = 0; s < p.splits; ++s) {
    const float ls = __ldcg(p.ws_lse + (unit0 + s) * kHeads + h);
    const float wgt = (M == -INFINITY || ls == -INFINITY) ? 0.f : exp2f(ls - M);
    W += wgt;
    const float4* src = reinterpret_cast<const float4*>(p.ws_o + ((unit0 + s) * kHeads + h) * kDvHalf + c0);
#pragma unroll
    for (int v = 0; v < 32; ++v) {
      const float4 x = __ldcg(src + v);
      acc[4 * v] = fmaf(wgt, x.x, acc[4 * v]);
      acc[4 * v + 1] = fmaf(wgt, x.y, acc[4 * v + 1]);
      acc[4 * v + 2] = fmaf(wgt, x.z, acc[4 * v + 2]);
      acc[4 * v + 3] = fmaf(wgt, x.w, acc[4 * v + 3]);
    }
  }
  if (h < p.H) {
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)t * p.H + h) * kDv + half * kDvHalf + c0);
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      uint4 w;
      w.x = pack_bf16(acc[8 * v] * inv, acc[8 * v + 1] * inv);
      w.y = pack_bf16(acc[8 * v + 2] * inv, acc[8 * v + 3] * inv);
      w.z = pack_bf16(acc[8 * v + 4] * inv, acc[8 * v + 5] * inv);
      w.w = pack_bf16(acc[8 * v + 6] * inv, acc[8 * v + 7] * inv);
      dst[v] = w;
    }
    if (half == 0 && c0 == 0 && p.lse)
      p.lse[(size_t)t * p.H + h] = W > 0.f ? (M + log2f(W)) * 0.69314718055994531f : -INFINITY;
  }
}

// CUDA-core variant (debug aid, selected by DSA_SFA_CUDA_CORE=1): one CTA per (token, head),
// direct two-pass softmax over the index set.
__global__ void __launch_bounds__(128) sfa_cuda_core_kernel(const Params p) {
  __shared__ float z[kMaxRows];
  __shared__ float red[4];
  const int t = blockIdx.x / p.H, h = blockIdx.x % p.H, tid = threadIdx.x;
  const int b = find_seq(p.q_start, p.B, t);
  const int L = p.seq_lens[b];
  const __nv_bfloat16* qh = p.q + ((size_t)t * p.H + h) * kDqk;
  float m = -INFINITY;
  for (int r = tid; r < p.K; r += 128) {
    const int j = p.idx[(size_t)t * p.K + r];
    float v = -INFINITY;
    if (j >= 0 && j < L) {
      const int pg = p.page_table[(size_t)b * p.max_pages + (j >> 6)];
      if (pg >= 0 && pg < p.num_pages) {
        const __nv_bfloat16* kv = p.kv + ((size_t)pg * 64 + (j & 63)) * kDqk;
        float d = 0.f;
        for (int c = 0; c < kDqk; ++c) d = fmaf(__bfloat162float(qh[c]), __bfloat162float(kv[c]), d);
        v = d * p.scale_log2;
      }
    }
    z[r] = v;
    m = fmaxf(m, v);
  }
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  float l = 0.f;
  for (int r = tid; r < p.K; r += 128) {
    const float e = (m == -INFINITY || z[r] == -INFINITY) ? 0.f : exp2f(z[r] - m);
    z[r] = e;
    l += e;
  }
  for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if ((tid & 31) == 0) red[tid >> 5] = l;
  __syncthreads();
  l = red[0] + red[1] + red[2] + red[3];
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int r = 0; r < p.K; ++r) {
    if (z[r] == 0.f) continue;
    const int j = p.idx[(size_t)t * p.K + r];
    const int pg = p.page_table[(size_t)b * p.max_pages + (j >> 6)];
    const __nv_bfloat16* kv = p.kv + ((size_t)pg * 64 + (j & 63)) * kDqk;
    for (int k = 0; k < 4; ++k) acc[k] = fmaf(z[r], __bfloat162float(kv[tid * 4 + k]), acc[k]);
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  for (int k = 0; k < 4; ++k) p.out[((size_t)t * p.H + h) * kDv + tid * 4 + k] = __float2bfloat16(acc[k] * inv);
  if (tid == 0 && p.lse) p.lse[(size_t)t * p.H + h] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
}

// ---------------------------------------------------------------- host side

struct Plan {
  int splits, rows_per;
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
  if (const char* e = std::getenv("DSA_SFA_SPLITS")) {
    const int s = std::atoi(e);
    if (s >= 1 && s <= 64) splits = s;
  }
  int rows_per = ((a.K + splits - 1) / splits + kNT - 1) / kNT * kNT;
  while (rows_per > kMaxRows) {  // K up to 2048 always fits one split
    ++splits;
    rows_per = ((a.K + splits - 1) / splits + kNT - 1) / kNT * kNT;
  }
  splits = (a.K + rows_per - 1) / rows_per;
  pl.splits = splits;
  pl.rows_per = rows_per;
  return pl;
}

static size_t ws_bytes(const dsa_sfa_args& a, const Plan& pl) {
  if (pl.splits <= 1) return 0;
  const size_t units = (size_t)a.n_q * 2 * pl.splits;
  size_t bytes = units * kHeads * kDvHalf * 4;   // partial o
  bytes += units * kHeads * 4;                    // partial lse
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
  if (need > 0) {
    const size_t units = (size_t)a.n_q * 2 * pl.splits;
    uint8_t* ws = reinterpret_cast<uint8_t*>(a.workspace);
    p.ws_o = reinterpret_cast<float*>(ws);
    p.ws_lse = reinterpret_cast<float*>(ws + units * kHeads * kDvHalf * 4);
    const size_t cnt_off = ((units * kHeads * kDvHalf * 4 + units * kHeads * 4) + 255) / 256 * 256;
    p.ws_count = reinterpret_cast<int*>(ws + cnt_off);
  } else {
    p.ws_o = nullptr;
    p.ws_lse = nullptr;
    p.ws_count = nullptr;
  }
  if (a.n_q == 0) return DSA_OK;

  const char* simple = std::getenv("DSA_SFA_CUDA_CORE");
  if (simple && simple[0] == '1') {
    sfa_cuda_core_kernel<<<a.n_q * a.H, 128, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "sfa (cuda-core): launch", err);
  }

  CUtensorMap tm_q, tm_kv;
  if (!encode_tmap_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kDqk, (uint64_t)a.n_q * a.H,
                      kDqk * 2, 64, kHeads, CU_TENSOR_MAP_SWIZZLE_128B, err))
    return DSA_ERR_CUDA;
  if (!encode_tmap_2d(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.kv_pool, kDqk,
                      (uint64_t)a.num_pages * 64, kDqk * 2, 64, 1, CU_TENSOR_MAP_SWIZZLE_128B, err))
    return DSA_ERR_CUDA;
  const int smem = Layout::total + 1024;
  cudaError_t e = cudaFuncSetAttribute(sfa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "sfa: set shared memory size", err);
  const unsigned grid = (unsigned)(a.n_q * 2 * pl.splits);
  if (std::getenv("DSA_VERBOSE"))
    std::fprintf(stderr, "[dsa] sfa %s splits=%d rows_per=%d grid=%u smem=%d\n",
                 prefill ? "prefill" : "decode", pl.splits, pl.rows_per, grid, smem);
  sfa_kernel<<<grid, kThreads, smem, stream>>>(tm_q, tm_kv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sfa: launch", err);
  return DSA_OK;
}

}  // namespace dsa
