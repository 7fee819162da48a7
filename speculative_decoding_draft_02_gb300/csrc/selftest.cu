// selftest.cu — failure detection without a fault.  Every device-side wait of
// the library is an mbarrier wait bounded in time; on expiry the kernel records
// DSPARK_ERR_TIMEOUT in the device status word and returns normally, so the
// context stays usable.  This entry point exercises exactly that path: one CTA
// waits, with the library's own bounded wait, on a barrier that no thread and
// no copy ever arrives on.
#include "tcgen05.cuh"

DSPARK_DECLARE_STATUS(s_status_selftest)

namespace {

__global__ void wait_on_silent_barrier(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);  // one arrival expected, none ever made
    abort = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, &abort, limit_ns))
    dspark_set_status(DSPARK_ERR_TIMEOUT);
}

}  // namespace

extern "C" int dspark_selftest_wait_timeout(uint64_t limit_ns, dspark_stream_t stream) {
  if (limit_ns == 0 || limit_ns > tc::WAIT_LIMIT_NS) return DSPARK_ERR_ARG;
  wait_on_silent_barrier<<<1, 32, 0, stream>>>(limit_ns);
  DSPARK_CHECK_LAUNCH();
  dspark_count_launches(1);
  return DSPARK_OK;
}

int dspark_status_selftest(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, s_status_selftest, sizeof(int)) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    cudaMemcpyToSymbol(s_status_selftest, &zero, sizeof(int));
  }
  return v;
}
