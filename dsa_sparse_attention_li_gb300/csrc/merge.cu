// merge.cu -- context-parallel indexer: merge of the shards' top-K candidates.
//
// Method: "Inference Optimization for Kimi K3.1 Pro: Decoding Architecture Evolution and Systems
// Engineering Practices", section 5 (hybrid parallelism: a local Top-K on each device before
// communication, so only K candidates per device cross the interconnect).  Each shard owns a
// disjoint range of a sequence's positions and selects its own top-K with dsa_li_topk (scores
// included); after the exchange every query's S*K candidates are merged here by the indexer's
// order (score descending, position ascending) and the first K are emitted ascending by position.
//
// One CTA per query: the candidates become 64-bit keys (order-preserving score key << 32 |
// ~position), a bitonic sort in shared memory orders them, and a second bitonic sort puts the
// first K positions in ascending order.  Exact and deterministic.
#include <climits>
#include <cstdio>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {
namespace merge {

constexpr int kThreads = 1024;
constexpr int kMaxCand = 16384;

// In-place bitonic sort of n (a power of two) entries of smem; descending when desc.
template <typename T>
DSA_DEV void bitonic(T* v, int n, bool desc) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += kThreads) {
        const int lo = 2 * stride * (i / stride) + (i % stride), hi = lo + stride;
        // the final merge (size == n) runs in the requested direction for every pair
        const bool d = ((lo & size) == 0) == desc;
        const T x = v[lo], y = v[hi];
        if (d ? (x < y) : (y < x)) {
          v[lo] = y;
          v[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kThreads)
    topk_merge_kernel(const dsa_topk_merge_args a, int ncand_pow2, int k_pow2) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  unsigned long long* key = reinterpret_cast<unsigned long long*>(smem_raw);
  uint32_t* pos = reinterpret_cast<uint32_t*>(key + ncand_pow2);
  __shared__ int valid;
  const int t = blockIdx.x, tid = threadIdx.x;
  if (tid == 0) valid = 0;
  for (int i = tid; i < ncand_pow2; i += kThreads) {
    unsigned long long k = 0ull;  // no candidate: sorts after every real one
    if (i < a.S * a.K_in) {
      const int s = i / a.K_in, r = i % a.K_in;
      const size_t at = ((size_t)s * a.n_q + t) * a.K_in + r;
      const int j = a.cand_idx[at];
      if (j >= 0) {
        const uint32_t p = (uint32_t)(j + a.shard_offset[s]);
        // score_key of a finite score is never 0, so real keys stay above "no candidate"
        k = ((unsigned long long)score_key(a.cand_score[at]) << 32) | (0xFFFFFFFFu - p);
      }
    }
    key[i] = k;
  }
  __syncthreads();
  bitonic(key, ncand_pow2, true);
  int mine = 0;
  for (int i = tid; i < k_pow2; i += kThreads) {
    uint32_t p = UINT_MAX;
    if (i < a.K && key[i] != 0ull) {
      p = 0xFFFFFFFFu - (uint32_t)(key[i] & 0xFFFFFFFFull);
      ++mine;
    }
    pos[i] = p;
  }
  atomicAdd(&valid, mine);
  __syncthreads();
  bitonic(pos, k_pow2, false);
  const int cnt = valid;
  for (int r = tid; r < a.K; r += kThreads)
    a.out_idx[(size_t)t * a.K + r] = r < cnt ? (int)pos[r] : -1;
  if (tid == 0 && a.out_cnt) a.out_cnt[t] = cnt;
}

// Largest b with q_start[b] <= t.
DSA_DEV int find_seq(const int* q_start, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (q_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Exclusive prefix sum over the 1024 threads of the block (wsum: 32 words of shared memory).
DSA_DEV uint32_t block_excl_scan(uint32_t v, uint32_t* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = wsum[lane];
    uint32_t z = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    wsum[lane] = z - w;
  }
  __syncthreads();
  const uint32_t r = wsum[warp] + x - v;
  __syncthreads();
  return r;
}

// Indexer over position units ("Inference Optimization for Kimi K3.1 Pro", section 5: a local
// Top-K per range of positions, then a merge of the candidates; here the ranges are units of one
// sequence on one GPU, so that long and short sequences of one batch spread evenly over the
// SMs).  One CTA per token whose sequence has more than one unit.  Its units' candidates (the
// exact top-K of disjoint, ascending position ranges, each list ascending with -1 padding) are
// concatenated in unit order, which keeps the positions ascending; a radix select over the
// order-preserving score keys (11, 11 and 10 bits) finds the K-th largest key and how many keys
// equal to it are taken, the lowest positions first; one ordered compaction writes the result.
// Runs as a programmatic dependent of the indexer: nothing is read before that grid completed.
__global__ void __launch_bounds__(kThreads)
    unit_merge_kernel(const UnitMergeArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t wsum[32];
  __shared__ uint32_t found[3];
  __shared__ int bsel[5];  // the token's sequence: index, matching ranges, length, range
  uint32_t* key = reinterpret_cast<uint32_t*>(smem_raw);   // [units * K] score keys, 0 = none
  int* pos = reinterpret_cast<int*>(key + a.units * a.K);  // [units * K]
  const int t = blockIdx.x, tid = threadIdx.x;
  if (tid == 0) {
    bsel[0] = -1;
    bsel[1] = 0;
  }
  __syncthreads();
  griddep_wait();
  // the token's sequence in one round of loads (every thread tests one sequence's range)
  for (int i = tid; i < a.B; i += kThreads) {
    const int s0 = a.q_start[i], s1 = a.q_start[i + 1], len = a.seq_lens[i];
    if (s0 <= t && t < s1) {
      atomicMax(&bsel[0], i);
      atomicAdd(&bsel[1], 1);
      bsel[2] = len;
      bsel[3] = s0;
      bsel[4] = s1;
    }
  }
  __syncthreads();
  int b = bsel[0], qs = bsel[3], n_b = bsel[4] - bsel[3], L = bsel[2];
  if (bsel[1] != 1) {  // q_start not increasing, or t outside it: the largest b with q_start[b] <= t
    b = find_seq(a.q_start, a.B, t);
    qs = a.q_start[b];
    n_b = a.q_start[b + 1] - qs;
    L = a.seq_lens[b];
  }
  // the indexer reported (and skipped) a sequence that fails these
  if (n_b <= 0 || L < n_b || L > a.units * a.span || L > a.max_pages * 64 || qs < 0 ||
      qs + n_b > a.n_q || n_b > a.groups * a.T || t - qs >= n_b)
    return;
  const int n_u = max(1, (L + a.span - 1) / a.span);
  if (n_u <= 1) return;  // the indexer wrote this token's result
  const int g = (t - qs) / a.T, tt = (t - qs) % a.T;
  const int ncand = n_u * a.K;
  // every load of a thread in flight at once: units x ceil(K / threads) <= 16 pairs; the keys
  // stay in registers for the three radix passes, the first of which is counted right here
  constexpr int kPer = kMaxCand / kThreads;
  uint32_t kr[kPer];
  {
    int jv[kPer];
    float sv[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + k * kThreads;
      jv[k] = -1;
      sv[k] = 0.f;
      if (i < ncand) {
        const int u = i / a.K, r = i - u * a.K;
        const size_t at = (((size_t)(b * a.groups + g) * a.units + u) * a.T + tt) * a.K + r;
        jv[k] = __ldcg(a.cand_idx + at);
        sv[k] = __ldcg(a.cand_score + at);
      }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + k * kThreads;
      // score_key of a finite score is never 0
      kr[k] = (i < ncand && jv[k] >= 0) ? score_key(sv[k]) : 0u;
      if (i < ncand) {
        key[i] = kr[k];
        pos[i] = jv[k];
      }
    }
  }
  // first pass (bits 31..21): the candidates are the units' top scores, so most share a few
  // high bins; the lanes of a warp that hit the same bin add their count with one atomic
  for (int i = tid; i < 2048; i += kThreads) hist[i] = 0u;
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    if (k * kThreads >= ncand) break;  // uniform
    const uint32_t bin = kr[k] != 0u ? kr[k] >> 21 : 0xffffffffu;
    const uint32_t peers = __match_any_sync(0xffffffffu, bin);
    if (kr[k] != 0u && (tid & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
  }
  __syncthreads();
  // Radix select of the K-th largest key: a pass finds the bin that holds it among the keys
  // that share the prefix fixed so far (thread i owns bins 2p + 1 and 2p with p = 1023 - i: the
  // exclusive prefix sum counts the keys in higher bins); passes 2 and 3 count only those keys,
  // from the registers.  The first pass also yields the number of valid candidates.
  uint32_t all = 0u, thr = 0u, need_eq = 0u;  // take keys > thr, and the first need_eq keys == thr
  {
    uint32_t prefix = 0u, pmask = 0u, need = (uint32_t)a.K;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const uint32_t bmask = pass == 2 ? 1023u : 2047u;
      if (pass > 0) {
        for (int i = tid; i < 2048; i += kThreads) hist[i] = 0u;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kPer; ++k)
          if (kr[k] != 0u && (kr[k] & pmask) == prefix) atomicAdd(&hist[(kr[k] >> shift) & bmask], 1u);
        __syncthreads();
      }
      const int pr = 1023 - tid;
      const uint32_t c_hi = hist[2 * pr + 1], c_lo = hist[2 * pr];
      const uint32_t above = block_excl_scan(c_hi + c_lo, wsum);
      if (pass == 0 && tid == kThreads - 1) found[1] = above + c_hi + c_lo;  // every key
      if (above < need && above + c_hi >= need) {
        found[0] = (uint32_t)(2 * pr + 1);
        found[1 + (pass == 0)] = need - above;
      } else if (above + c_hi < need && above + c_hi + c_lo >= need) {
        found[0] = (uint32_t)(2 * pr);
        found[1 + (pass == 0)] = need - above - c_hi;
      }
      __syncthreads();
      if (pass == 0) {
        all = found[1];
        if (all <= (uint32_t)a.K) break;  // uniform: every candidate is taken
        need = found[2];
      } else {
        need = found[1];
      }
      prefix |= found[0] << shift;
      pmask |= bmask << shift;
      __syncthreads();
    }
    if (all > (uint32_t)a.K) {
      thr = prefix;
      need_eq = need;
    }
  }
  const uint32_t cnt = min(all, (uint32_t)a.K);
  // ordered compaction: thread i takes the contiguous run [i * per, (i + 1) * per)
  const int per = (ncand + kThreads - 1) / kThreads;
  const int c0 = min(ncand, tid * per), c1 = min(ncand, c0 + per);
  uint32_t eq = 0;
  for (int i = c0; i < c1; ++i) eq += (key[i] == thr && thr != 0u);
  uint32_t eq_before = block_excl_scan(eq, wsum);
  uint32_t take = 0;
  for (int i = c0; i < c1; ++i) {
    const uint32_t k = key[i];
    if (k > thr) {
      ++take;
    } else if (k == thr && thr != 0u) {
      if (eq_before < need_eq) ++take;
      ++eq_before;
    }
  }
  uint32_t at = block_excl_scan(take, wsum);
  eq_before -= eq;  // back to this run's first tie
  int* out = a.out_idx + (size_t)t * a.K;
  float* osc = a.out_score ? a.out_score + (size_t)t * a.K : nullptr;
  for (int i = c0; i < c1; ++i) {
    const uint32_t k = key[i];
    bool sel = k > thr;
    if (k == thr && thr != 0u) sel = eq_before++ < need_eq;
    if (sel) {
      out[at] = pos[i];
      if (osc) osc[at] = key_score(k);
      ++at;
    }
  }
  for (int r = (int)cnt + tid; r < a.K; r += kThreads) {
    out[r] = -1;
    if (osc) osc[r] = -INFINITY;
  }
  if (tid == 0 && a.out_cnt) a.out_cnt[t] = (int)cnt;
}

}  // namespace merge

dsa_status launch_topk_merge(const dsa_topk_merge_args& a, cudaStream_t stream, std::string& err) {
  using namespace merge;
  if (a.n_q == 0) return DSA_OK;
  int nc = 1, kp = 1;
  while (nc < a.S * a.K_in) nc <<= 1;
  while (kp < a.K) kp <<= 1;
  const int smem = nc * 8 + kp * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "topk_merge: set shared memory size", err);
  topk_merge_kernel<<<a.n_q, kThreads, smem, stream>>>(a, nc, kp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "topk_merge: launch", err);
  return DSA_OK;
}

dsa_status launch_unit_merge(const UnitMergeArgs& a, cudaStream_t stream, std::string& err) {
  using namespace merge;
  if (a.n_q == 0) return DSA_OK;
  if ((long long)a.units * a.K > kMaxCand) {
    err = "li_topk: " + std::to_string(a.units) + " units x K exceed the merge capacity";
    return DSA_ERR_UNSUPPORTED;
  }
  const int smem = a.units * a.K * 8;
  cudaError_t e = cudaFuncSetAttribute(unit_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e, "li_topk: set unit merge shared memory size", err);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_q);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, unit_merge_kernel, a);
  if (e != cudaSuccess) return cuda_fail(e, "li_topk: unit merge launch", err);
  return DSA_OK;
}

}  // namespace dsa
