// Diagnostic kernel for the device-side failure path: a bounded mbarrier wait that cannot
// complete (nothing ever arrives on the barrier) gives up after the device wait limit,
// raises the timeout bit of the status word, and the kernel then releases its tensor
// memory the way the tensor-core kernels do after a timeout (commit-drain, dealloc) and
// returns, so the context stays usable.  Nothing faults, traps or hangs.
#include "tc.cuh"
#include "tc_ptx.cuh"

namespace dpk {

__global__ void __launch_bounds__(64, 1) selftest_wait_kernel(unsigned* status, unsigned long long* waited_ns) {
  __shared__ uint64_t never;   // count 1; no thread or copy ever arrives
  __shared__ uint64_t drain;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&never, 1);
    ptx::mbar_init(&drain, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (threadIdx.x < 32) ptx::tmem_alloc(&tslot, 32);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tslot;
  const uint64_t t0 = ptx::globaltimer();
  if (threadIdx.x < 32) {
    const bool w = ptx::mbar_wait(&never, 0, &abort_flag, status);   // runs out: abort + timeout status
    (void)__all_sync(0xffffffffu, w);
  }
  __syncthreads();
  if (*(volatile int*)&abort_flag && threadIdx.x == 0) {
    ptx::umma_commit(&drain);   // arrives once every MMA issued so far (none) has completed
    ptx::mbar_wait_drain(&drain, 0);
  }
  if (threadIdx.x == 0 && waited_ns) *waited_ns = ptx::globaltimer() - t0;
  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 32);
  }
}

}  // namespace dpk

namespace dph {
cudaError_t launch_selftest_wait(unsigned* status, unsigned long long* waited_ns, cudaStream_t s) {
  launch_plain(dpk::selftest_wait_kernel, 1, 64, 0, s, status, waited_ns);
  return cudaGetLastError();
}
}  // namespace dph
