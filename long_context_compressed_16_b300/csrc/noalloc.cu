// csa_index_topk_noalloc: the indexer + top-k call without a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the moment they need to select entries: code
// that runs inside a host callback or a custom allocator hook (where calling cudaMalloc would
// re-enter the allocator or synchronise the device), runtimes that hand out only pre-planned
// tensors, and plug-ins whose host gives them input and output buffers but no allocator.  For
// them the scratch space (status word + fp32 score rows) lives in one fixed array in device
// memory that the library module declares.  Every GPU that loads the library holds the array
// until the process exits; its size is CSA_NOALLOC_SCRATCH_BYTES.
//
// The host side never dereferences the array's name: in host code it is only a stand-in, and
// the real device address comes from cudaGetSymbolAddress, once per device, with that device
// current.  The address is cached, so later calls make no CUDA call beyond the launches.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_index_scratch[CSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's copy of g_index_scratch (looked up on first use).
csa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_index_scratch) != cudaSuccess || p == nullptr) return CSA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CSA_OK;
}

}  // namespace

extern "C" csa_status csa_index_topk_noalloc(const csa_index_desc* desc, const void* qI, const float* w,
                                             const void* kI, const float* kI_scale, const int32_t* q_pos,
                                             int32_t* idx_out, float* score_out, csa_stream_t stream) {
  const size_t need = csa_index_topk_workspace(desc);
  if (need == 0) return CSA_ERR_INVALID_ARG;
  if (need > CSA_NOALLOC_SCRATCH_BYTES) return CSA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const csa_status st = scratch_address(&scratch);
  if (st != CSA_OK) return st;
  // csa_index_topk clears the status word itself and writes every score it later reads, so the
  // previous call's contents of the array need no clearing here.
  return csa_index_topk(desc, qI, w, kI, kI_scale, q_pos, idx_out, score_out, scratch,
                        CSA_NOALLOC_SCRATCH_BYTES, stream);
}
