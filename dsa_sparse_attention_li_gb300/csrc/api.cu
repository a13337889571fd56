// api.cu -- the C ABI (include/dsa.h): host-side validation, status codes, per-thread error
// text, TMA descriptor encoding and device-property caching.  No entry point allocates memory,
// synchronises, or keeps a pointer after it returns.
#include <cudaTypedefs.h>

#include <mutex>
#include <string>
#include <unordered_set>
#include <vector>

#include "dsa_internal.h"

namespace {

thread_local std::string g_last_error;

dsa_status fail(dsa_status s, const std::string& why) {
  g_last_error = why;
  return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace dsa {

#ifdef DSA_TEST_HOOKS
int g_test_stall = 0;
#endif

void set_last_error(const std::string& why) { g_last_error = why; }

bool device_info(DeviceInfo& info, std::string& err) {
  static std::mutex mu;
  static std::vector<DeviceInfo> cache(64);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    err = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
    return false;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < (int)cache.size() && cache[dev].device == dev) {
    info = cache[dev];
    return true;
  }
  DeviceInfo d;
  d.device = dev;
  e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) {
    err = std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e);
    return false;
  }
  if (dev >= 0 && dev < (int)cache.size()) cache[dev] = d;
  info = d;
  return true;
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                    uint32_t box_outer, CUtensorMapSwizzle swizzle, std::string& err) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  if (!fn) {
    err = "cuTensorMapEncodeTiled is not available from the driver";
    return false;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

}  // namespace dsa

extern "C" {

const char* dsa_status_string(dsa_status s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE_CHECK: return "DSA_ERR_DEVICE_CHECK";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
  }
  return "DSA_ERR_UNKNOWN";
}

const char* dsa_last_error(void) { return g_last_error.c_str(); }

int dsa_abi_version(void) { return DSA_ABI_VERSION; }

size_t dsa_page_bytes(dsa_dtype dtype, int rows, int dim) {
  if (rows < 0 || dim < 0) return 0;
  const size_t elt = dtype == DSA_BF16 ? 2 : ((dtype == DSA_FP8_E4M3 || dtype == DSA_MXFP8_E4M3) ? 1 : 0);
  return elt * (size_t)rows * (size_t)dim;
}

dsa_status dsa_page_table_validate(const int32_t* pt, int B, int max_pages, const int32_t* seq_lens,
                                   int page_size, int num_pages, int require_unique) {
  g_last_error.clear();
  if (!pt || !seq_lens || B <= 0 || max_pages <= 0 || page_size <= 0 || num_pages <= 0)
    return fail(DSA_ERR_INVALID_ARG, "page_table_validate: null pointer or non-positive size");
  std::vector<uint8_t> used(require_unique ? (size_t)num_pages : 0, 0);
  for (int b = 0; b < B; ++b) {
    const long long L = seq_lens[b];
    if (L < 0) return fail(DSA_ERR_INVALID_ARG, "seq_lens[" + std::to_string(b) + "] < 0");
    const long long np = (L + page_size - 1) / page_size;
    if (np > max_pages)
      return fail(DSA_ERR_INVALID_ARG, "sequence " + std::to_string(b) + " needs " +
                                           std::to_string(np) + " pages > max_pages");
    for (long long p = 0; p < np; ++p) {
      const int id = pt[(size_t)b * max_pages + p];
      if (id < 0 || id >= num_pages)
        return fail(DSA_ERR_INVALID_ARG, "page_table[" + std::to_string(b) + "][" +
                                             std::to_string(p) + "] = " + std::to_string(id) +
                                             " out of [0, num_pages)");
      if (require_unique) {
        if (used[id])
          return fail(DSA_ERR_INVALID_ARG, "page " + std::to_string(id) + " used twice");
        used[id] = 1;
      }
    }
  }
  return DSA_OK;
}

dsa_status dsa_li_topk(const dsa_li_args* a, dsa_stream_t stream) {
  g_last_error.clear();
  if (!a) return fail(DSA_ERR_INVALID_ARG, "li_topk: args is NULL");
  if (a->B <= 0 || a->n_q < 0 || a->K <= 0 || a->max_pages <= 0 || a->num_pages <= 0 ||
      a->H_I <= 0 || a->d_I <= 0)
    return fail(DSA_ERR_INVALID_ARG, "li_topk: non-positive size");
  if (a->dtype != DSA_BF16 && a->dtype != DSA_FP8_E4M3 && a->dtype != DSA_MXFP8_E4M3)
    return fail(DSA_ERR_INVALID_ARG, "li_topk: unknown dtype");
  if (a->n_q == 0) return DSA_OK;
  if (!a->q || !a->w || !a->k_pool || !a->page_table || !a->seq_lens || !a->q_start || !a->out_idx)
    return fail(DSA_ERR_INVALID_ARG, "li_topk: null device pointer");
  if (a->dtype == DSA_FP8_E4M3 && (!a->q_scale || !a->k_scale))
    return fail(DSA_ERR_INVALID_ARG, "li_topk: FP8 needs q_scale and k_scale");
  if (a->dtype == DSA_MXFP8_E4M3 &&
      (!a->q_sf || !a->k_sf || ((reinterpret_cast<uintptr_t>(a->q_sf) | reinterpret_cast<uintptr_t>(a->k_sf)) & 3u) != 0))
    return fail(DSA_ERR_INVALID_ARG, "li_topk: MXFP8 needs 4-byte aligned q_sf and k_sf");
  if (a->max_seq_len <= 0 || a->max_q_per_seq <= 0 || a->max_q_per_seq > a->n_q)
    return fail(DSA_ERR_INVALID_ARG, "li_topk: max_seq_len / max_q_per_seq out of range");
  if ((long long)a->max_seq_len > (long long)a->max_pages * a->page_size)
    return fail(DSA_ERR_INVALID_ARG, "li_topk: max_seq_len exceeds max_pages * page_size");
  if (!aligned16(a->q) || !aligned16(a->k_pool))
    return fail(DSA_ERR_INVALID_ARG, "li_topk: q and k_pool must be 16-byte aligned");
  if (a->page_size != 64) return fail(DSA_ERR_UNSUPPORTED, "li_topk: page_size must be 64");
  if (a->K > 2048) return fail(DSA_ERR_UNSUPPORTED, "li_topk: K > 2048");
  if (a->max_seq_len > 131072) return fail(DSA_ERR_UNSUPPORTED, "li_topk: max_seq_len > 131072");
  if (a->workspace != nullptr && (reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
    return fail(DSA_ERR_INVALID_ARG, "li_topk: workspace must be 256-byte aligned");
  std::string err;
  const dsa_status s = dsa::launch_li_topk(*a, reinterpret_cast<cudaStream_t>(stream), err);
  if (s != DSA_OK) g_last_error = err;
  return s;
}

size_t dsa_li_workspace_bytes(const dsa_li_args* a) {
  if (!a || a->B <= 0 || a->K <= 0 || a->max_seq_len <= 0 || a->max_q_per_seq <= 0) return 0;
  return dsa::li_workspace_bytes(*a);
}

static dsa_status sfa_common(const dsa_sfa_args* a, bool prefill, dsa_stream_t stream) {
  g_last_error.clear();
  const char* name = prefill ? "sfa_prefill" : "sfa_decode";
  if (!a) return fail(DSA_ERR_INVALID_ARG, std::string(name) + ": args is NULL");
  if (a->B <= 0 || a->n_q < 0 || a->H <= 0 || a->K <= 0 || a->max_pages <= 0 || a->num_pages <= 0)
    return fail(DSA_ERR_INVALID_ARG, std::string(name) + ": non-positive size");
  if (!(a->softmax_scale > 0.f) || a->softmax_scale != a->softmax_scale)
    return fail(DSA_ERR_INVALID_ARG, std::string(name) + ": softmax_scale must be positive");
  if (a->n_q == 0) return DSA_OK;
  if (!a->q || !a->kv_pool || !a->page_table || !a->seq_lens || !a->q_start || !a->idx || !a->out)
    return fail(DSA_ERR_INVALID_ARG, std::string(name) + ": null device pointer");
  if (!aligned16(a->q) || !aligned16(a->kv_pool) || !aligned16(a->out))
    return fail(DSA_ERR_INVALID_ARG, std::string(name) + ": q, kv_pool, out must be 16-byte aligned");
  if (a->d_qk != 576 || a->d_v != 512)
    return fail(DSA_ERR_UNSUPPORTED, std::string(name) + ": d_qk must be 576 and d_v 512");
  if (a->page_size != 64) return fail(DSA_ERR_UNSUPPORTED, std::string(name) + ": page_size must be 64");
  if (a->kv_dtype != DSA_BF16 && a->kv_dtype != DSA_FP8_E4M3)
    return fail(DSA_ERR_UNSUPPORTED, std::string(name) + ": kv_dtype must be BF16 or FP8_E4M3");
  if (a->H > 128) return fail(DSA_ERR_UNSUPPORTED, std::string(name) + ": H > 128");
  if (a->K > 2048) return fail(DSA_ERR_UNSUPPORTED, std::string(name) + ": K > 2048");
  std::string err;
  const dsa_status s = dsa::launch_sfa(*a, prefill, reinterpret_cast<cudaStream_t>(stream), err);
  if (s != DSA_OK) g_last_error = err;
  return s;
}

size_t dsa_sfa_workspace_bytes(const dsa_sfa_args* a) {
  if (!a || a->n_q <= 0 || a->K <= 0) return 0;
  return dsa::sfa_workspace_bytes(*a);
}

dsa_status dsa_sfa_decode(const dsa_sfa_args* a, dsa_stream_t stream) {
  return sfa_common(a, false, stream);
}

dsa_status dsa_sfa_prefill(const dsa_sfa_args* a, dsa_stream_t stream) {
  return sfa_common(a, true, stream);
}

dsa_status dsa_topk_merge(const dsa_topk_merge_args* a, dsa_stream_t stream) {
  g_last_error.clear();
  if (!a) return fail(DSA_ERR_INVALID_ARG, "topk_merge: null args");
  if (a->S <= 0 || a->n_q < 0 || a->K_in <= 0 || a->K <= 0)
    return fail(DSA_ERR_INVALID_ARG, "topk_merge: non-positive size");
  if ((long long)a->S * a->K_in > 16384 || a->K > 16384)
    return fail(DSA_ERR_UNSUPPORTED, "topk_merge: S * K_in and K must be at most 16384");
  if (a->n_q > 0 && (!a->cand_idx || !a->cand_score || !a->shard_offset || !a->out_idx))
    return fail(DSA_ERR_INVALID_ARG, "topk_merge: null device pointer");
  std::string err;
  const dsa_status s = dsa::launch_topk_merge(*a, reinterpret_cast<cudaStream_t>(stream), err);
  if (s != DSA_OK) g_last_error = err;
  return s;
}

static dsa_status prolog_check(const dsa_prolog_args* a, bool pointers) {
  if (!a) return fail(DSA_ERR_INVALID_ARG, "indexer_prolog: null args");
  if (a->n_q < 0 || a->B <= 0 || a->d_q <= 0 || a->d_model <= 0 || a->max_pages <= 0 ||
      a->num_pages <= 0)
    return fail(DSA_ERR_INVALID_ARG, "indexer_prolog: non-positive size");
  if (a->H_I != 64 || a->d_I != 128 || a->page_size != 64)
    return fail(DSA_ERR_UNSUPPORTED, "indexer_prolog: needs H_I 64, d_I 128, page_size 64");
  if (a->dtype != DSA_MXFP8_E4M3 && a->dtype != DSA_BF16)
    return fail(DSA_ERR_UNSUPPORTED, "indexer_prolog: dtype must be MXFP8_E4M3 or BF16");
  if (a->d_q % 8 || a->d_model % 8)
    return fail(DSA_ERR_UNSUPPORTED, "indexer_prolog: d_q and d_model must be multiples of 8");
  if (!pointers) return DSA_OK;  // sizes only (workspace query)
  if (!a->xq || !a->x || !a->w_q || !a->w_k || !a->w_w || !a->ln_gamma || !a->ln_beta ||
      !a->page_table || !a->seq_lens || !a->q_start || !a->q_out || !a->w_out || !a->k_pool ||
      (a->dtype == DSA_MXFP8_E4M3 && (!a->q_sf || !a->k_sf)))
    return fail(DSA_ERR_INVALID_ARG, "indexer_prolog: null device pointer");
  if (!aligned16(a->xq) || !aligned16(a->x) || !aligned16(a->w_q) || !aligned16(a->w_k) ||
      !aligned16(a->w_w))
    return fail(DSA_ERR_INVALID_ARG, "indexer_prolog: inputs and weights must be 16-byte aligned");
  return DSA_OK;
}

size_t dsa_prolog_workspace_bytes(const dsa_prolog_args* a) {
  if (prolog_check(a, false) != DSA_OK) return 0;
  return dsa::prolog_workspace_bytes(*a);
}

dsa_status dsa_indexer_prolog(const dsa_prolog_args* a, dsa_stream_t stream) {
  g_last_error.clear();
  const dsa_status c = prolog_check(a, true);
  if (c != DSA_OK) return c;
  std::string err;
  const dsa_status s = dsa::launch_prolog(*a, reinterpret_cast<cudaStream_t>(stream), err);
  if (s != DSA_OK) g_last_error = err;
  return s;
}

dsa_status dsa_cache_write(void* pool, float* scale_pool, int num_pages, int page_size, int dim,
                           int elem_bytes, const int32_t* page_table, int max_pages, int B,
                           const int32_t* seq, const int32_t* pos, const void* rows,
                           const float* row_scales, int n_rows, int32_t* status,
                           dsa_stream_t stream) {
  g_last_error.clear();
  if (n_rows < 0 || num_pages <= 0 || page_size <= 0 || dim <= 0 || max_pages <= 0 || B <= 0)
    return fail(DSA_ERR_INVALID_ARG, "cache_write: non-positive size");
  if (elem_bytes != 1 && elem_bytes != 2)
    return fail(DSA_ERR_INVALID_ARG, "cache_write: elem_bytes must be 1 or 2");
  if ((dim * elem_bytes) % 16 != 0)
    return fail(DSA_ERR_UNSUPPORTED, "cache_write: row bytes must be a multiple of 16");
  if (n_rows == 0) return DSA_OK;
  if (!pool || !page_table || !seq || !pos || !rows)
    return fail(DSA_ERR_INVALID_ARG, "cache_write: null device pointer");
  if (!aligned16(pool) || !aligned16(rows))
    return fail(DSA_ERR_INVALID_ARG, "cache_write: pool and rows must be 16-byte aligned");
  if ((scale_pool == nullptr) != (row_scales == nullptr))
    return fail(DSA_ERR_INVALID_ARG, "cache_write: scale_pool and row_scales go together");
  std::string err;
  const dsa_status s = dsa::launch_cache_write(pool, scale_pool, num_pages, page_size, dim,
                                               elem_bytes, page_table, max_pages, B, seq, pos,
                                               rows, row_scales, n_rows, status,
                                               reinterpret_cast<cudaStream_t>(stream), err);
  if (s != DSA_OK) g_last_error = err;
  return s;
}

#ifdef DSA_TEST_HOOKS
// Test build only (libdsa_testhooks.so; include/dsa_testhooks.h).
void dsa_test_inject_stall(int kernel) { dsa::g_test_stall = kernel; }
#endif

}  // extern "C"
