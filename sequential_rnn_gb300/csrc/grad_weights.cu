// Helpers around the weight gradients of the head-wise cells:
//   * h0 -> bf16, so the dR contraction can read h_{-1} = h0 as its first K rows
//     (the contraction itself, dR[h] = sum_{t,b} h_{t-1}^T dG_t, runs on the
//     tcgen05 tensor cores in tc_gemm.cu);
//   * db[h] = sum_{t,b} dG_t, summed from the per-batch-slice partials the
//     reverse kernel leaves in the workspace.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace srnn {
namespace {

__global__ void h0_to_bf16_kernel(const float* __restrict__ h0, __nv_bfloat16* __restrict__ out,
                                  int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    out[i] = __float2bfloat16_rn(h0 ? h0[i] : 0.f);
}

__global__ void db_reduce_kernel(const float* __restrict__ part, float* __restrict__ db,
                                 int nslices, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int k = 0; k < nslices; ++k) s += part[(size_t)k * n + i];
    db[i] = s;
  }
}

}  // namespace

int launch_h0_to_bf16(const float* h0, void* out, int n, cudaStream_t s) {
  const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
  h0_to_bf16_kernel<<<blocks > 0 ? blocks : 1, 256, 0, s>>>(h0, static_cast<__nv_bfloat16*>(out), n);
  return (int)cudaGetLastError();
}

int launch_db_reduce(const float* part, float* db, int nslices, int n, cudaStream_t s) {
  const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
  db_reduce_kernel<<<blocks > 0 ? blocks : 1, 256, 0, s>>>(part, db, nslices, n);
  return (int)cudaGetLastError();
}

}  // namespace srnn
