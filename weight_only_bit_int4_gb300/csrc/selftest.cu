// selftest.cu -- a self-test of the bounded pipeline waits, without any fault.
//
// Every mbarrier wait of the library gives up after a wall-clock limit, records
// Q4MM_DEVERR_WAIT_TIMEOUT, sets the CTA's abort flag so the other roles unwind, and lets
// the copies already in flight land before the CTA exits.  This kernel runs that sequence on
// purpose with a short limit: one thread starts a real bulk copy (its barrier completes),
// then waits on a barrier that nothing arrives on, times out and aborts; it then waits for
// its copy in flight, as the pipelines do when they unwind.  A second warp waits on another
// barrier that nothing arrives on and leaves when it sees the abort flag.  Nothing traps.
#include "tc_common.cuh"

namespace q4mm {

Q4MM_DEFINE_ERROR_READER(read_errors_selftest)

namespace {

__global__ void __launch_bounds__(64) wait_timeout_selftest_kernel(const void *src16, unsigned long long limit_ns) {
  __shared__ __align__(128) uint8_t buf[16];
  __shared__ __align__(8) uint64_t bars[3];   // 0: the copy, 1 and 2: never completed
  __shared__ int abort_flag;
  const uint32_t b0 = smem_u32(&bars[0]), b1 = smem_u32(&bars[1]), b2 = smem_u32(&bars[2]);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 3; ++i) tc::mbar_init(smem_u32(&bars[i]), 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  volatile int *abort = &abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_arrive_expect_tx(b0, 16u);
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 16, [%2];" ::"r"(
                     smem_u32(buf)),
                 "l"(src16), "r"(b0)
                 : "memory");
    tc::mbar_wait(b1, 0u, abort, 200, limit_ns);   // times out: sets the error bit and *abort
    volatile int dummy = 0;
    tc::mbar_wait(b0, 0u, &dummy, 200);            // the copy in flight lands before exit
  } else if (threadIdx.x == 32) {
    tc::mbar_wait(b2, 0u, abort, 200);             // leaves on the abort flag
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(const void *src16, unsigned long long limit_ns, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 64, 0, s>>>(src16, limit_ns);
  return cudaGetLastError();
}

}  // namespace q4mm
