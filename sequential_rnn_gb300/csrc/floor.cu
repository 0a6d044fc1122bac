// Sync-floor kernel: the per-step synchronisation of a forward launch with
// nothing else (no loads, no math).  Same grid, block size and cluster shape
// as the forward it stands for, and the same barrier kind:
//   * fp32 path: one CTA barrier per step;
//   * bf16, one CTA per head slice: one named barrier over the compute warps;
//   * bf16 cluster: each compute warp st.async's 4 bytes into every cluster
//     CTA's mbarrier-tracked buffer and all threads wait for the phase.
// time / T of this kernel is the "sync floor" term of the per-step roofline.
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace srnn {
namespace {

__global__ void floor_cta_kernel(int T, int nbar) {
  for (int t = 0; t < T; ++t)
    for (int b = 0; b < nbar; ++b) __syncthreads();
}

__global__ void floor_named_kernel(int T, int NW) {
  const int warp = threadIdx.x >> 5;
  if (warp < NW) {
    for (int t = 0; t < T; ++t) bar_sync(1, NW * 32);
  }
}

__global__ void floor_cluster_kernel(int T, int CS, int NW, unsigned long long tlim, int* status) {
  __shared__ __align__(16) uint32_t buf[2][64];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t b0 = smem_u32(&bars[0]);
  const uint32_t tx = (uint32_t)(NW * CS * 4);
  if (tid == 0) {
    mbar_init(b0, 1);
    mbar_init(b0 + 8, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    if (T >= 2) mbar_arrive_expect_tx(b0 + 8, tx);
    if (T >= 3) mbar_arrive_expect_tx(b0, tx);
  }
  cluster_sync();
  if (warp < NW) {
    for (int t = 0; t < T; ++t) {
      if (t > 0) {
        const uint32_t bar = b0 + 8 * (t & 1);
        const uint32_t par = ((t - 1) >> 1) & 1;
        const uint64_t t0 = globaltimer_ns();
        bool ok = true;
        while (!mbar_try_wait(bar, par)) {
          if (globaltimer_ns() - t0 > tlim) {
            atomicOr(status, kStatusTimeout);
            ok = false;
            break;
          }
        }
        if (!ok) break;
        if (tid == 0 && t + 1 <= T - 2) mbar_arrive_expect_tx(bar, tx);
      }
      __syncwarp();
      if (t + 1 < T && lane == 0) {
        const uint32_t la = smem_u32(&buf[(t + 1) & 1][warp]);
        const uint32_t lb = b0 + 8 * ((t + 1) & 1);
        for (int r = 0; r < CS; ++r) st_async_b32(mapa(la, r), (uint32_t)t, mapa(lb, r));
      }
    }
  }
  cluster_sync();
}

}  // namespace

int launch_sync_floor(const LaunchInfo& li, int T, int* status, cudaStream_t s) {
  if (li.kernel_id >= 1000) {  // fp32 path: one CTA barrier per step
    floor_cta_kernel<<<li.grid, li.threads, 0, s>>>(T, 1);
    return (int)cudaGetLastError();
  }
  const int NW = li.threads / 32;  // bf16 forward: compute warps only
  if (li.cluster <= 1) {
    floor_named_kernel<<<li.grid, li.threads, 0, s>>>(T, NW);
    return (int)cudaGetLastError();
  }
  if (NW > 64) return (int)cudaErrorInvalidValue;
  if (li.cluster > 8) {
    cudaError_t e =
        cudaFuncSetAttribute(floor_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return (int)e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(li.grid);
  cfg.blockDim = dim3(li.threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = li.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, floor_cluster_kernel, T, li.cluster, NW,
                                 2000000000ull, status);
}

}  // namespace srnn
