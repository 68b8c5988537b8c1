// Self-test of the failure detection every kernel of the library relies on:
// a bounded mbarrier wait that runs out records MLA_DEV_TIMEOUT, raises the
// abort flag of its CTA and of the other CTAs of its cluster, and returns, so
// the kernel ends instead of hanging the GPU.
//
// The kernel waits on barriers that nothing ever arrives at.  In a two-CTA
// cluster, CTA 1 waits with the caller's short limit and CTA 0 with the
// library's full limit; CTA 0 must come back as soon as CTA 1 gives up,
// through the propagated abort flag.  Each CTA reports how long its wait took.
#include "kernels.cuh"

namespace mla {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(int32_t* status, long long* elapsed_ns,
                                                           unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t n = cluster_size();
  const uint32_t rank = cluster_rank();
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (n > 1) cluster_sync(); else __syncthreads();
  if (threadIdx.x == 0) {
    // In a cluster only the last CTA uses the short limit.
    const uint64_t limit = (n > 1 && rank + 1 < n) ? kWaitLimitNs : limit_ns;
    const uint64_t t0 = globaltimer();
    const bool ok = mbar_wait(smem_u32(&bar), 0, status, &abort_flag, limit);
    elapsed_ns[blockIdx.x] = ok ? -1 : static_cast<long long>(globaltimer() - t0);
  }
  // No CTA leaves while another may still write its abort flag.
  if (n > 1) cluster_sync(); else __syncthreads();
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(int32_t* status, long long* elapsed_ns, uint64_t limit_ns,
                                         int cluster, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bounded_wait_kernel, status, elapsed_ns,
                            static_cast<unsigned long long>(limit_ns));
}

}  // namespace mla
