// dsa_internal.h -- host-side declarations shared by the C-ABI front end and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <string>

#include "dsa.h"

namespace dsa {

// Launchers: arguments are already validated by the front end (api.cu).
dsa_status launch_li_topk(const dsa_li_args& a, cudaStream_t stream, std::string& err);
dsa_status launch_sfa(const dsa_sfa_args& a, bool prefill, cudaStream_t stream, std::string& err);
size_t sfa_workspace_bytes(const dsa_sfa_args& a);
dsa_status launch_prolog(const dsa_prolog_args& a, cudaStream_t stream, std::string& err);
dsa_status launch_topk_merge(const dsa_topk_merge_args& a, cudaStream_t stream, std::string& err);

// Indexer over position units: workspace bytes dsa_li_topk needs (0 when no sequence is split).
size_t li_workspace_bytes(const dsa_li_args& a);
// Merge of the units' top-K candidates of every token whose sequence was split (merge.cu): unit u
// of token group g of sequence b left its candidates of token tt at slot
// ((b * groups + g) * units + u) * T + tt of cand_idx / cand_score ([slots][K]).
struct UnitMergeArgs {
  int B, n_q, K, T, groups, units;
  int span;       // positions a cluster covers: a sequence of L positions has ceil(L / span) units
  int max_pages;  // (the indexer's validity bound on L)
  const int* seq_lens;
  const int* q_start;
  int* cand_idx;
  float* cand_score;
  int* out_idx;
  int* out_cnt;
  float* out_score;
};
dsa_status launch_unit_merge(const UnitMergeArgs& a, cudaStream_t stream, std::string& err);
size_t prolog_workspace_bytes(const dsa_prolog_args& a);
dsa_status launch_cache_write(void* pool, float* scale_pool, int num_pages, int page_size, int dim,
                              int elem_bytes, const int32_t* page_table, int max_pages, int B,
                              const int32_t* seq, const int32_t* pos, const void* rows,
                              const float* row_scales, int n_rows, int32_t* status,
                              cudaStream_t stream, std::string& err);

// 2-D tiled TMA descriptor over a row-major [outer][inner] array (inner contiguous).
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner, uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                    uint32_t box_outer, CUtensorMapSwizzle swizzle, std::string& err);

#ifdef DSA_TEST_HOOKS
// Test build only: which kernel's first CTA makes one of its waits wait on a barrier that nothing
// arrives on (0 none, 1 li_topk, 2 sparse attention); set by dsa_test_inject_stall().
extern int g_test_stall;
#endif

// Sets the calling thread's dsa_last_error() text.
void set_last_error(const std::string& why);

// Device properties of the current device (cached per device).
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int smem_optin = 0;   // max dynamic shared memory per block
  int smem_per_sm = 0;  // shared memory per multiprocessor
  int cc_major = 0, cc_minor = 0;
};
bool device_info(DeviceInfo& info, std::string& err);

inline dsa_status cuda_fail(cudaError_t e, const char* what, std::string& err) {
  err = std::string(what) + ": " + cudaGetErrorString(e);
  return DSA_ERR_CUDA;
}

}  // namespace dsa
