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
// the real device address comes from cudaGetSymbolAddress with the device current.  That address
// belongs to one CUDA context (the module is loaded once per context), so the cache is keyed by
// the context's process-unique ID (cuCtxGetId): a caller's own context, or the new primary
// context after cudaDeviceReset, gets its own lookup instead of another context's address.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_index_scratch[CSA_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name, int version) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(f);
}

constexpr int kCacheSlots = 64;
struct ScratchSlot {
  unsigned long long ctx_id;
  void* addr;
};
std::mutex g_scratch_mu;
ScratchSlot g_slots[kCacheSlots] = {};
int g_next_slot = 0;

// Device address of g_index_scratch in the calling thread's current context.  The first call in
// a context looks the address up; later calls in that context find it in the cache.
csa_status scratch_address(void** out) {
  static const CtxGetCurrentFn get_ctx = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 12000);
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
  if (!get_ctx || !get_id) return CSA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
    // no context bound to this thread yet: cudaSetDevice binds (and initialises) the device's
    // primary context, the one the runtime would use for the launches
    if (cudaSetDevice(dev) != cudaSuccess) return CSA_ERR_CUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return CSA_ERR_CUDA;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return CSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  for (const ScratchSlot& s : g_slots) {
    if (s.addr != nullptr && s.ctx_id == id) {
      *out = s.addr;
      return CSA_OK;
    }
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_index_scratch) != cudaSuccess || p == nullptr) return CSA_ERR_CUDA;
  g_slots[g_next_slot] = ScratchSlot{id, p};
  g_next_slot = (g_next_slot + 1) % kCacheSlots;
  *out = p;
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
  // The kernels write every score they later read, so the previous call's scores need no
  // clearing.  The status word does: csa_index_topk only ever sets it, so it is zeroed on the
  // stream before each call (the caller cannot read it; see the header).
  if (cudaMemsetAsync(scratch, 0, 8, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return CSA_ERR_CUDA;
  return csa_index_topk(desc, qI, w, kI, kI_scale, q_pos, idx_out, score_out, scratch,
                        CSA_NOALLOC_SCRATCH_BYTES, stream);
}
