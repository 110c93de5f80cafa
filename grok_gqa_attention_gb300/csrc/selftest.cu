// Self-test of the bounded-wait machinery every pipelined kernel relies on.
//
// One CTA, two warps, two mbarriers that nothing ever arrives on. Warp 0 waits
// with the caller's short limit and gives up: it records GROK_DEV_TIMEOUT and
// raises the CTA's abort flag. Warp 1 waits with a limit 1000 times longer and
// must leave through that abort flag well before its own limit. The kernel
// then returns normally, which is what the real kernels do after a timeout.
#include "common.cuh"
#include "host.cuh"

namespace grok {

__global__ void __launch_bounds__(64) selftest_wait_kernel(int32_t* status, int32_t* flags, long long limit) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &abort_flag;
  bool ok;
  if (warp == 0)
    ok = mbar_wait_for(&bars[0], 0, abort, status, limit);
  else
    ok = mbar_wait_for(&bars[1], 0, abort, status, limit * 1000);
  ok = __all_sync(0xffffffffu, ok);
  if (lane == 0) flags[warp] = ok ? 1 : 2;  // 2 = gave up (timeout or abort)
}

}  // namespace grok

using namespace grok;

extern "C" grok_status grok_selftest_bounded_wait(int32_t* dev_status, int32_t* flags, long long limit_cycles,
                                                  void* stream) {
  if (!dev_status || !flags) return fail(GROK_ERR_INVALID_ARG, "grok_selftest_bounded_wait: null pointer");
  if (limit_cycles < 1 || limit_cycles > 4000000000LL)
    return fail(GROK_ERR_INVALID_ARG, "grok_selftest_bounded_wait: limit must be in [1, 4e9] cycles");
  int sms = 0;
  grok_status st = device_sm_count(&sms);
  if (st != GROK_OK) return st;
  selftest_wait_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(dev_status, flags, limit_cycles);
  return check_launch("selftest_wait");
}
