// ds_topk_select_static: the exact top-k of ds_topk_select for callers that
// cannot allocate device memory.
//
// Some callers of a decode step have no way to obtain a workspace: a plugin
// that runs inside a host framework which owns every device allocation and
// hands it only the tensors of the call, or a real-time serving thread that
// may not block on an allocator's lock. For them this entry point takes its
// scratch from a fixed array compiled into the library instead of from a
// caller-provided workspace, and allocates nothing.
//
// The array lives in device global memory on every GPU that loads the
// library, for as long as the process runs. Its size caps the problem: a
// (shape, k) whose top-k scratch exceeds DS_TOPK_STATIC_SCRATCH_BYTES is
// rejected with DS_ERR_WORKSPACE before anything is launched.
#include <cuda_runtime.h>

#include <atomic>

#include "ds_sparse.h"

// One copy per device. In host code `g_topk_static_scratch` only names a
// host-side shadow symbol, not device memory: its device address must be
// fetched with cudaGetSymbolAddress on each device.
static __device__ __align__(256) unsigned char g_topk_static_scratch[DS_TOPK_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

// Device address of the scratch array on the current device, looked up on the
// first call made with that device current (nullptr on failure). Two threads
// that make their first call at once both look it up and store the same
// address; the atomics make that well defined. A cudaDeviceReset invalidates
// the cached address (the header says so).
void* static_scratch() {
  static std::atomic<void*> ptrs[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = ptrs[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_topk_static_scratch) != cudaSuccess) return nullptr;
    ptrs[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace

extern "C" ds_status ds_topk_select_static(const ds_shape* shape, const float* scores, const int32_t* seq_lens,
                                           int k, int32_t* idx, ds_stream_t stream) {
  const size_t need = ds_topk_workspace_bytes(shape, k);
  if (need == 0) return ds_topk_select(shape, scores, seq_lens, k, idx, nullptr, 0, stream);  // argument error
  if (need > static_cast<size_t>(DS_TOPK_STATIC_SCRATCH_BYTES)) return DS_ERR_WORKSPACE;
  void* scratch = static_scratch();
  if (!scratch) return DS_ERR_CUDA;
  // ds_topk_select needs no initialised scratch (it only spills candidate
  // lists there), so leftovers of the previous call do no harm.
  return ds_topk_select(shape, scores, seq_lens, k, idx, scratch, DS_TOPK_STATIC_SCRATCH_BYTES, stream);
}
