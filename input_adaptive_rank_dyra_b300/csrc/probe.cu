// Self-test of the forward's failure path: one CTA waits, with the same bounded mbarrier wait
// that every role of the GEMM engine uses, on a barrier that nothing arrives on. The wait
// gives up after the given limit, counts itself in the status word and the kernel returns,
// so the host sees DYRA_ERR_TIMEOUT and the context stays usable. No TMA or MMA is in flight
// while the wait runs, and nothing else touches the barrier.
#include "kernels.cuh"
#include "ptx.cuh"

namespace dyra {

namespace {

__global__ void __launch_bounds__(32) bounded_wait_probe_kernel(int *status,
                                                                unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);      // one arrival expected; none comes
    ptx::mbar_init_fence();
  }
  __syncwarp();
  if (threadIdx.x == 0) ptx::mbar_wait(b, 0, status + 1, limit_ns);
}

}  // namespace

cudaError_t launch_bounded_wait_probe(int *status, unsigned long long limit_ns, cudaStream_t s) {
  bounded_wait_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace dyra
