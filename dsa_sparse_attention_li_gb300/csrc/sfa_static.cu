// sfa_static.cu -- dsa_sfa_decode_static: sparse-attention decode for callers that cannot
// allocate device memory.
//
// Who needs it: code whose device memory is planned and owned by a host framework that hands an
// operator only its inputs and outputs (no per-call workspace, no allocator handle), and code
// running where an allocation is not allowed at all (a path that must never block on, or fail
// in, the memory allocator).  Such callers cannot provide the split-merge workspace that
// dsa_sfa_decode asks for.
//
// How: the workspace lives in the file-scope device array below, of a fixed capacity
// (DSA_SFA_STATIC_SCRATCH_BYTES); every GPU that loads this library holds it until the process
// exits.  Host code never passes the array's name to a kernel -- in host code that name is only a
// host-side stand-in for the symbol -- it asks the runtime for the device address once per
// device.  The call then forwards to dsa_sfa_decode with that address as the workspace, so the
// arithmetic and the result are exactly those of dsa_sfa_decode.
#include <mutex>
#include <string>

#include "dsa_internal.h"

namespace {

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) unsigned char g_sfa_scratch[DSA_SFA_STATIC_SCRATCH_BYTES];

struct ScratchSlot {
  bool ready = false;
  void* ptr = nullptr;
};

std::mutex g_mu;
ScratchSlot g_slots[64];

}  // namespace

extern "C" dsa_status dsa_sfa_decode_static(const dsa_sfa_args* a, dsa_stream_t stream) {
  if (!a) {
    dsa::set_last_error("sfa_decode_static: args is NULL");
    return DSA_ERR_INVALID_ARG;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    dsa::set_last_error(std::string("sfa_decode_static: cudaGetDevice: ") + cudaGetErrorString(e));
    return DSA_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) {
    dsa::set_last_error("sfa_decode_static: device ordinal out of range");
    return DSA_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  {
    // One-time set-up per device, with that device current: the scratch array's device address.
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_slots[dev].ready) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_sfa_scratch);
      if (e != cudaSuccess) {
        dsa::set_last_error(std::string("sfa_decode_static: cudaGetSymbolAddress: ") +
                            cudaGetErrorString(e));
        return DSA_ERR_CUDA;
      }
      g_slots[dev].ptr = p;
      g_slots[dev].ready = true;
    }
    scratch = g_slots[dev].ptr;
  }
  const size_t need = dsa_sfa_workspace_bytes(a);
  if (need > (size_t)DSA_SFA_STATIC_SCRATCH_BYTES) {
    dsa::set_last_error("sfa_decode_static: these arguments need " + std::to_string(need) +
                        " bytes of scratch, above the fixed capacity of " +
                        std::to_string((size_t)DSA_SFA_STATIC_SCRATCH_BYTES) +
                        " bytes (use dsa_sfa_decode with a caller workspace)");
    return DSA_ERR_UNSUPPORTED;
  }
  if (need > 0) {
    // The split-merge arrival counters (the tail of the workspace) must start at zero; the
    // kernel returns them to zero, but a call that stopped early could have left them set.
    const size_t counters = ((size_t)a->n_q * 2 * sizeof(int) + 255) / 256 * 256;
    e = cudaMemsetAsync(static_cast<unsigned char*>(scratch) + (need - counters), 0, counters,
                        reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
      dsa::set_last_error(std::string("sfa_decode_static: clearing counters: ") +
                          cudaGetErrorString(e));
      return DSA_ERR_CUDA;
    }
  }
  dsa_sfa_args b = *a;
  b.workspace = scratch;
  b.workspace_bytes = (size_t)DSA_SFA_STATIC_SCRATCH_BYTES;
  return dsa_sfa_decode(&b, stream);
}
