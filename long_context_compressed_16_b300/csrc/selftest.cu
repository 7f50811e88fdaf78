// Failure-path diagnostic.  Every wait inside the library's kernels is bounded: a wait that is
// never satisfied gives up after its limit, records CSA_ERR_TIMEOUT in the workspace status word
// and lets the kernel return, so the CUDA context stays usable.  This call runs that path on
// purpose with a wait that nothing can complete (an mbarrier that no thread arrives on).
#include "common.cuh"
#include "tc.cuh"

namespace csa {
namespace {

__global__ void __launch_bounds__(32) k_selftest_wait(int32_t* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  grid_dep_wait();
  grid_dep_launch();
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_barrier_init();
    const uint64_t t0 = tc::globaltimer_ns();
    if (!tc::mbar_wait(&bar, 0, nullptr, limit_ns)) {
      const uint64_t us = (tc::globaltimer_ns() - t0) / 1000u;
      report_error(status, CSA_ERR_TIMEOUT, static_cast<int32_t>(us > 0x7FFFFFFFull ? 0x7FFFFFFFull : us));
    }
  }
}

}  // namespace
}  // namespace csa

extern "C" csa_status csa_selftest_bounded_wait(void* ws, size_t ws_bytes, int64_t limit_ns, csa_stream_t stream) {
  if (!ws || ws_bytes < csa::kStatusBytes) return CSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 15u) != 0) return CSA_ERR_INVALID_ARG;
  if (limit_ns < 1000 || limit_ns > 2000000000LL) return CSA_ERR_INVALID_ARG;
  const cudaError_t e = csa::launch_k(csa::k_selftest_wait, dim3(1), dim3(32), 0,
                                      reinterpret_cast<cudaStream_t>(stream), static_cast<int32_t*>(ws),
                                      static_cast<unsigned long long>(limit_ns));
  csa::note_launches(1);
  return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
