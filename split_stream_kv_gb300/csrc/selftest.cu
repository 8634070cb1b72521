// selftest.cu -- a check of the bounded-wait pattern every asynchronous-copy
// wait of the library follows (mbarrier try-wait in a loop on the global
// timer, give up after a limit, report instead of hanging), run on a barrier
// that nothing completes, and (arrive == 2) of the verification kernel's own
// wait and abort word (attn_tc.cu).  Used by the tests to show that such a
// wait ends and leaves the context usable; it faults and traps nothing.
#include "common.cuh"
#include "internal.h"
#include "lynx.h"

namespace lynx {

// attn_tc.cu: the verification kernel's wait and its abort word
cudaError_t launch_tc_wait_selftest(uint64_t limit_ns, unsigned int* status, cudaStream_t stream);

namespace {

__global__ void wait_selftest_kernel(uint64_t limit_ns, int arrive, unsigned int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (arrive && threadIdx.x == 0)
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(&bar)) : "memory");
  bool ok = mbar_try_wait(&bar, 0);
  const uint64_t t0 = global_ns();
  while (!ok && global_ns() - t0 < limit_ns) ok = mbar_try_wait(&bar, 0);
  __syncthreads();
  if (threadIdx.x == 0) *status = ok ? 1u : 2u;
}

}  // namespace
}  // namespace lynx

using namespace lynx;

extern "C" int lynx_wait_selftest(uint64_t limit_ns, int arrive, unsigned int* status,
                                  void* stream) {
  if (!status) return report_error(LYNX_EINVAL, "null pointer");
  if (limit_ns == 0 || limit_ns > 1000000000ull)
    return report_error(LYNX_EINVAL, "limit_ns must be in (0, 1e9]");
  cudaError_t e;
  if (arrive == 2) {
    e = launch_tc_wait_selftest(limit_ns, status, static_cast<cudaStream_t>(stream));
  } else {
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, arrive, status);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return report_error(LYNX_ECUDA, cudaGetErrorString(e));
  return LYNX_OK;
}
