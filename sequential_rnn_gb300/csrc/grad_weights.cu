// Weight gradients of the head-wise cells after the reverse recurrence.
//
//   dR[h] = sum_{t,b} h_{t-1}[b,h,:]^T dG_t[b,h,:]      (h_{-1} = h0)
//   db[h] = sum_{t,b} dG_t[b,h,:]
// with dG the gradient of the recurrent preactivation (h @ R + b): dWx for the
// LSTM and sLSTM; for the GRU it differs from dWx on the n block (r * dn~).
//
// dR is one dense contraction per head over K = T*B rows: the only true GEMM
// of the path.  Tensor cores (mma.sync bf16 -> fp32) on 128x128 output tiles,
// K streamed in 32-row chunks through a 3-stage cp.async ring; both operands
// are read in their natural row-major layouts (h rows of Dh, dG rows of G*Dh)
// and transposed on the fly by ldmatrix.trans.  db is summed from the
// per-batch-slice partials the reverse kernel leaves in the workspace.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace srnn {
namespace {

constexpr int BM = 128, BN = 128, BK = 32, NSTG = 3;
constexpr int PITCH = BM * 2 + 16;                 // bytes per smem row (17 chunks: odd)
constexpr int STAGE = 2 * BK * PITCH;              // A then B
constexpr int SMEM = NSTG * STAGE;

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}

// grid: (ceil(G*Dh/BN), ceil(Dh/BM), NH); 256 threads = 8 warps as 2 (M) x 4 (N),
// each warp a 64 x 32 tile = 4 x 4 mma m16n8.
__global__ void __launch_bounds__(256) dR_gemm_kernel(const __nv_bfloat16* __restrict__ h_seq,
                                                      const __nv_bfloat16* __restrict__ h0b,
                                                      const __nv_bfloat16* __restrict__ dWx,
                                                      float* __restrict__ dR, int T, int B, int NH,
                                                      int Dh, int G) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int GD = G * Dh;
  const int head = blockIdx.z;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 2, wn = warp & 3;  // warp tile origin: (wm*64, wn*32)
  const int R = T * B;
  const int nchunks = (R + BK - 1) / BK;
  const uint32_t sb = smem_u32(smem);

  // each thread copies 2 A chunks and 2 B chunks of 16 bytes per stage
  auto load_stage = [&](int kc, int stg) {
    const uint32_t sA = sb + stg * STAGE, sB = sA + BK * PITCH;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = tid + i * 256;  // 0..511: row = c / 16, 16-byte column = c % 16
      const int row = c >> 4, col8 = (c & 15) * 8;
      const int r = kc * BK + row;
      // A: h_{t-1} row of this head, units m0 + col8 ..
      const bool va = r < R && m0 + col8 < Dh;
      const __nv_bfloat16* srcA = h0b;
      if (va) {
        srcA = r < B ? h0b + ((size_t)r * NH + head) * Dh + m0 + col8
                     : h_seq + ((size_t)(r - B) * NH + head) * Dh + m0 + col8;
      }
      cp_async16_zfill(sA + row * PITCH + col8 * 2, srcA, va);
      // B: dG row, gate columns n0 + col8 ..
      const bool vb = r < R && n0 + col8 < GD;
      const __nv_bfloat16* srcB = vb ? dWx + ((size_t)r * NH + head) * GD + n0 + col8 : dWx;
      cp_async16_zfill(sB + row * PITCH + col8 * 2, srcB, vb);
    }
  };

  float acc[4][4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[a][b][q] = 0.f;

#pragma unroll
  for (int s = 0; s < NSTG - 1; ++s) {
    if (s < nchunks) load_stage(s, s);
    cp_async_commit();
  }
  // ldmatrix.trans lane addressing (see mma fragment layouts):
  //   A (stored [k][m]): matrix q = lane>>3 -> (m +8*(q&1), k +8*(q>>1))
  //   B (stored [k][n]): matrix q -> (k +8*(q&1), n +8*(q>>1))
  const int lr = lane & 7, lq = lane >> 3;
  for (int kc = 0; kc < nchunks; ++kc) {
    cp_async_wait<NSTG - 2>();
    __syncthreads();
    {
      const int nk = kc + NSTG - 1;
      if (nk < nchunks) load_stage(nk, nk % NSTG);
      cp_async_commit();
    }
    const uint32_t sA = sb + (kc % NSTG) * STAGE, sB = sA + BK * PITCH;
#pragma unroll
    for (int ks = 0; ks < BK / 16; ++ks) {
      uint32_t af[4][4], bfm[2][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int m = wm * 64 + mt * 16 + 8 * (lq & 1);
        const int k = ks * 16 + lr + 8 * (lq >> 1);
        ldmatrix_x4_trans(af[mt], sA + k * PITCH + m * 2);
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int n = wn * 32 + np * 16 + 8 * (lq >> 1);
        const int k = ks * 16 + lr + 8 * (lq & 1);
        ldmatrix_x4_trans(bfm[np], sB + k * PITCH + n * 2);
      }
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          mma_bf16_16816(acc[mt][nt], af[mt], bfm[nt >> 1][2 * (nt & 1)], bfm[nt >> 1][2 * (nt & 1) + 1]);
    }
  }
  cp_async_wait<0>();
  // epilogue: fp32 pairs
  float* out = dR + (size_t)head * Dh * GD;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int m = m0 + wm * 64 + mt * 16 + (lane >> 2) + 8 * half;
        const int n = n0 + wn * 32 + nt * 8 + 2 * (lane & 3);
        if (m < Dh && n < GD)
          *reinterpret_cast<float2*>(out + (size_t)m * GD + n) =
              make_float2(acc[mt][nt][2 * half], acc[mt][nt][2 * half + 1]);
      }
}

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

int launch_grad_weights(const void* h_seq, const void* h0_bf16, const void* dWx, float* dR, int T,
                        int B, int NH, int Dh, int G, cudaStream_t s) {
  if (G != 3 && G != 4) return (int)cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(dR_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return (int)e;
  dim3 grid((G * Dh + BN - 1) / BN, (Dh + BM - 1) / BM, NH);
  dR_gemm_kernel<<<grid, 256, SMEM, s>>>(static_cast<const __nv_bfloat16*>(h_seq),
                                         static_cast<const __nv_bfloat16*>(h0_bf16),
                                         static_cast<const __nv_bfloat16*>(dWx), dR, T, B, NH, Dh, G);
  return (int)cudaGetLastError();
}

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
