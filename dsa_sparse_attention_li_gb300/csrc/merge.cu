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

}  // namespace dsa
