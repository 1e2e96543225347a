// Self-test of the failure path the tensor-core kernels share: a pipeline wait
// (mbar_wait, the bounded mbarrier wait of every producer, MMA and epilogue loop)
// on a barrier that nothing arrives on must give up after its limit, raise
// MOE_DEV_TIMEOUT in the caller's error word and return, leaving the context usable.
#include "tc.cuh"

namespace moe {
namespace {

__global__ void wait_timeout_kernel(int32_t *err, uint64_t timeout_ns, int32_t *waited) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(&bar), 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = tc::globaltimer();
    const bool ok = tc::mbar_wait(tc::smem_u32(&bar), 0, &abort_flag, err, timeout_ns);
    // report how long the wait lasted (ms) and that it gave up
    if (waited) *waited = ok ? -1 : (int32_t)((tc::globaltimer() - t0) / 1000000ull);
  }
}

}  // namespace
}  // namespace moe

MOE_API moe_status_t moe_selftest_wait_timeout(int32_t *err, int64_t timeout_ns, int32_t *waited_ms,
                                               moe_stream_t stream) {
  if (!err || timeout_ns < 1000 || timeout_ns > 100000000) return MOE_ERR_INVALID_ARG;
  moe::wait_timeout_kernel<<<1, 32, 0, moe::as_cuda(stream)>>>(err, (uint64_t)timeout_ns, waited_ms);
  return moe::launch_status();
}
