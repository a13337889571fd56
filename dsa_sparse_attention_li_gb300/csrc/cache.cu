// cache.cu -- paged-cache helpers: scatter new rows (keys of the indexer cache or latent rows of
// the attention cache) into their pages through the page table.
//
// The pages describe both caches as paged ("Day0 Inference Adaptation ... CANN", section 3.1:
// the indexer reads the paged K cache, SFA reads the main attention KV at the selected indices;
// "Inference Optimization for Kimi K3.1 Pro ...", section 2: on-demand in-page addressing).
#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {

// One warp per row: 16-byte vector copies of the row, plus its scale for FP8 key caches.
__global__ void __launch_bounds__(256) cache_write_kernel(
    uint8_t* pool, float* scale_pool, int num_pages, int page_size, int row_bytes,
    const int32_t* page_table, int max_pages, int B, const int32_t* seq, const int32_t* pos,
    const uint8_t* rows, const float* row_scales, int n_rows, int32_t* status) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= n_rows) return;
  const int b = seq[warp], j = pos[warp];
  if (b < 0 || b >= B || j < 0 || j / page_size >= max_pages) {
    if (lane == 0) report(status, kStatusDeviceCheck);
    return;
  }
  const int pg = page_table[(size_t)b * max_pages + j / page_size];
  if (pg < 0 || pg >= num_pages) {
    if (lane == 0) report(status, kStatusDeviceCheck);
    return;
  }
  const size_t dst_row = (size_t)pg * page_size + j % page_size;
  const uint4* src = reinterpret_cast<const uint4*>(rows + (size_t)warp * row_bytes);
  uint4* dst = reinterpret_cast<uint4*>(pool + dst_row * row_bytes);
  for (int v = lane; v < row_bytes / 16; v += 32) dst[v] = src[v];
  if (lane == 0 && scale_pool && row_scales) scale_pool[dst_row] = row_scales[warp];
}

dsa_status launch_cache_write(void* pool, float* scale_pool, int num_pages, int page_size, int dim,
                              int elem_bytes, const int32_t* page_table, int max_pages, int B,
                              const int32_t* seq, const int32_t* pos, const void* rows,
                              const float* row_scales, int n_rows, int32_t* status,
                              cudaStream_t stream, std::string& err) {
  if (n_rows == 0) return DSA_OK;
  const int row_bytes = dim * elem_bytes;
  const int threads = 256;
  const long long blocks = ((long long)n_rows * 32 + threads - 1) / threads;
  cache_write_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
      reinterpret_cast<uint8_t*>(pool), scale_pool, num_pages, page_size, row_bytes, page_table,
      max_pages, B, seq, pos, reinterpret_cast<const uint8_t*>(rows), row_scales, n_rows, status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "cache_write: launch", err);
  return DSA_OK;
}

}  // namespace dsa
