// fp32 forward of the head-wise recurrence: the precision reference path.
//
// One CTA per (head, batch slice of up to 8 rows).  Thread k (0 <= k < G*Dh)
// owns gate row k of the head and keeps column k of R[h] in registers for the
// whole time loop (FlashRNN blog page, register-caching paragraph: R pinned
// in registers inside a persistent kernel).  Per step:
//   1. rec[b][k] = sum_j h_{t-1}[b][j] * R[j][k] + bias[k]   (fp32 FMA, h from smem)
//   2. barrier
//   3. each (b, j) cell thread applies the gates with accurate expf/tanhf,
//      updates its state and writes h_t to shared memory and h_seq
//   4. barrier
// Wx_t rows are prefetched NSTG steps ahead with cp.async into a smem ring.
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace srnn {

namespace {
constexpr int kNB = 8;    // batch rows per CTA
constexpr int kNSTG = 4;  // Wx ring depth (steps in flight)

__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + expf(-x)); }

template <int CELL, int DH>
__global__ void __launch_bounds__(256, 1) fwd_f32_kernel(const FwdParams p) {
  constexpr int G = CELL == kGRU ? 3 : 4;
  constexpr int GD = G * DH;
  constexpr int EPT = (kNB * DH + GD - 1) / GD;  // cells per thread
  __shared__ __align__(16) float hs[kNB][DH];
  __shared__ __align__(16) float rec[kNB][GD];
  __shared__ __align__(16) float xs[kNSTG][kNB][GD];

  const int k = threadIdx.x;
  const int T = p.T, B = p.B, NH = p.NH;
  const int head = blockIdx.x / p.nbslices, bslice = blockIdx.x % p.nbslices;
  const int b0 = bslice * kNB;
  const int nb = min(kNB, B - b0);
  const float* Wx = static_cast<const float*>(p.Wx);
  const float* Rh = static_cast<const float*>(p.R) + (size_t)head * DH * GD;
  float* hseq = static_cast<float*>(p.h_seq);

  float rcol[DH];
#pragma unroll
  for (int j = 0; j < DH; ++j) rcol[j] = Rh[(size_t)j * GD + k];
  const float bk = p.bias ? p.bias[(size_t)head * GD + k] : 0.f;

  float st_c[EPT], st_n[EPT], st_m[EPT], st_h[EPT];
#pragma unroll
  for (int q = 0; q < EPT; ++q) {
    const int e = k + q * GD;
    const int b = e / DH, j = e % DH;
    const bool ok = e < nb * DH;
    const size_t si = ((size_t)(b0 + b) * NH + head) * DH + j;
    st_h[q] = (ok && p.h0) ? p.h0[si] : 0.f;
    st_c[q] = (ok && p.c0) ? p.c0[si] : 0.f;
    st_n[q] = (ok && p.n0) ? p.n0[si] : 0.f;
    st_m[q] = (ok && p.m0) ? p.m0[si] : 0.f;
  }
  for (int e = k; e < kNB * DH; e += GD) {
    const int b = e / DH, j = e % DH;
    hs[b][j] = (b < nb && p.h0) ? p.h0[((size_t)(b0 + b) * NH + head) * DH + j] : 0.f;
  }
  for (int b = nb; b < kNB; ++b)
    for (int s = 0; s < kNSTG; ++s) xs[s][b][k] = 0.f;

  auto issue = [&](int t) {
    if (t < T) {
      const int s = t % kNSTG;
      for (int b = 0; b < nb; ++b)
        cp_async4(smem_u32(&xs[s][b][k]), Wx + (((size_t)t * B + b0 + b) * NH + head) * GD + k);
    }
    cp_async_commit();
  };
#pragma unroll 1
  for (int t = 0; t < kNSTG - 1; ++t) issue(t);
  __syncthreads();

#pragma unroll 1
  for (int t = 0; t < T; ++t) {
    issue(t + kNSTG - 1);
    cp_async_wait<kNSTG - 1>();
    const int s = t % kNSTG;
    // 1. recurrent preactivation for gate row k, all batch rows
    float acc[kNB];
#pragma unroll
    for (int b = 0; b < kNB; ++b) acc[b] = 0.f;
#pragma unroll
    for (int j = 0; j < DH; j += 4) {
#pragma unroll
      for (int b = 0; b < kNB; ++b) {
        const float4 hv = *reinterpret_cast<const float4*>(&hs[b][j]);
        acc[b] = fmaf(hv.x, rcol[j], acc[b]);
        acc[b] = fmaf(hv.y, rcol[j + 1], acc[b]);
        acc[b] = fmaf(hv.z, rcol[j + 2], acc[b]);
        acc[b] = fmaf(hv.w, rcol[j + 3], acc[b]);
      }
    }
#pragma unroll
    for (int b = 0; b < kNB; ++b) rec[b][k] = acc[b] + bk;
    __syncthreads();
    // 3. cell update
#pragma unroll
    for (int q = 0; q < EPT; ++q) {
      const int e = k + q * GD;
      if (e >= nb * DH) continue;
      const int b = e / DH, j = e % DH;
      float h;
      if (CELL == kLSTM) {
        const float ig = sigm(rec[b][j] + xs[s][b][j]);
        const float fg = sigm(rec[b][DH + j] + xs[s][b][DH + j]);
        const float zg = tanhf(rec[b][2 * DH + j] + xs[s][b][2 * DH + j]);
        const float og = sigm(rec[b][3 * DH + j] + xs[s][b][3 * DH + j]);
        st_c[q] = fg * st_c[q] + ig * zg;
        h = og * tanhf(st_c[q]);
      } else if (CELL == kGRU) {
        const float rg = sigm(xs[s][b][j] + rec[b][j]);
        const float zg = sigm(xs[s][b][DH + j] + rec[b][DH + j]);
        const float ng = tanhf(xs[s][b][2 * DH + j] + rg * rec[b][2 * DH + j]);
        h = (1.f - zg) * ng + zg * st_h[q];
      } else {
        const float pi = rec[b][j] + xs[s][b][j];
        const float pf = rec[b][DH + j] + xs[s][b][DH + j];
        const float pz = rec[b][2 * DH + j] + xs[s][b][2 * DH + j];
        const float po = rec[b][3 * DH + j] + xs[s][b][3 * DH + j];
        const float mn = fmaxf(pf + st_m[q], pi);
        const float ig = expf(pi - mn);
        const float fg = expf(pf + st_m[q] - mn);
        st_c[q] = fg * st_c[q] + ig * tanhf(pz);
        st_n[q] = fg * st_n[q] + ig;
        st_m[q] = mn;
        h = sigm(po) * (st_c[q] / st_n[q]);
      }
      st_h[q] = h;
      hs[b][j] = h;
      hseq[(((size_t)t * B + b0 + b) * NH + head) * DH + j] = h;
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  if (T > 0) {
#pragma unroll
    for (int q = 0; q < EPT; ++q) {
      const int e = k + q * GD;
      if (e >= nb * DH) continue;
      const int b = e / DH, j = e % DH;
      const size_t si = ((size_t)(b0 + b) * NH + head) * DH + j;
      if (p.hT) p.hT[si] = st_h[q];
      if (p.cT && CELL != kGRU) p.cT[si] = st_c[q];
      if (p.nT && CELL == kSLSTM) p.nT[si] = st_n[q];
      if (p.mT && CELL == kSLSTM) p.mT[si] = st_m[q];
    }
  }
}

template <int CELL, int DH>
int launch_t(const FwdParams& p, cudaStream_t s, bool query_only, LaunchInfo* info) {
  constexpr int G = CELL == kGRU ? 3 : 4;
  const int grid = p.NH * p.nbslices;
  if (info) *info = LaunchInfo{grid, G * DH, 1, kNB, 0, 1000 + CELL * 100 + DH};
  if (query_only) return 0;
  fwd_f32_kernel<CELL, DH><<<grid, G * DH, 0, s>>>(p);
  return (int)cudaGetLastError();
}

template <int CELL>
int launch_cell(const FwdParams& p, int Dh, cudaStream_t s, bool q, LaunchInfo* info) {
  switch (Dh) {
    case 16: return launch_t<CELL, 16>(p, s, q, info);
    case 32: return launch_t<CELL, 32>(p, s, q, info);
    case 64: return launch_t<CELL, 64>(p, s, q, info);
    default: return (int)cudaErrorInvalidValue;
  }
}
}  // namespace

int launch_fwd_f32(const FwdParams& p, int cell, int Dh, cudaStream_t s, bool query_only,
                   LaunchInfo* info) {
  if (cell == kLSTM) return launch_cell<kLSTM>(p, Dh, s, query_only, info);
  if (cell == kGRU) return launch_cell<kGRU>(p, Dh, s, query_only, info);
  return launch_cell<kSLSTM>(p, Dh, s, query_only, info);
}

}  // namespace srnn
