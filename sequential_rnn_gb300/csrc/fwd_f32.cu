// fp32 forward of the head-wise recurrence: the precision reference path.
//
// One CTA per (head, batch row): the rows of a batch are independent
// recurrences (FlashRNN blog page, head-wise paragraph: heads -- and batch
// rows -- map to separate thread blocks), so each step's latency chain is one
// row's.  Thread (lane 4 (j % 8) + g of warp j / 8) owns gate row g*Dh + j and
// keeps column g*Dh + j of R[h] in registers for the whole time loop (blog
// page, register-caching paragraph), so the G gates of hidden unit j sit in
// adjacent lanes of one warp.  Per step:
//   1. the thread's dot product over h_{t-1}: packed fp32 FMAs (fma.rn.f32x2,
//      each lane of the pair rounded as a scalar fma) in eight chains, h read
//      from shared memory as broadcast float4;
//   2. each thread activates its own gate with accurate tanhf (a sigmoid as
//      1/2 + tanh(x/2)/2, so the four lanes of a unit run the same code), and
//      the unit's lane 4 (j % 8) gathers the G values by shuffles, applies the
//      cell, updates its fp32 state and writes h_t to shared memory and h_seq
//      (GRU: the reset gate reaches the n lane by one shuffle first; sLSTM:
//      the stabilised exponential gates stay on the cell lane, which holds m);
//   3. one CTA barrier (h is double-buffered by step parity).
// (A split of each dot product over four threads -- 1024 threads for
// Dh = 64 -- ran 990 ns per step: a barrier of 32 warps alone takes ~160 ns.)
// Wx rows are streamed PD steps ahead into a shared-memory ring with 16-byte
// cp.async issued by the first G*Dh/4 threads; each thread waits for its own
// copies before the barrier that precedes their first read, and a slot is
// refilled only after the barrier that follows its last read.
#include <cuda_runtime.h>

#include "check.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace srnn {

namespace {
constexpr int kPD = 4;  // Wx ring depth (steps)

// two fp32 FMAs in one instruction: (a.x b.x + c.x, a.y b.y + c.y), each rounded once
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  return (unsigned long long)__float_as_uint(lo) | ((unsigned long long)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float lo2(unsigned long long v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(unsigned long long v) { return __uint_as_float((uint32_t)(v >> 32)); }

template <int CELL, int DH>
__global__ void __launch_bounds__(DH * 4, 1) fwd_f32_kernel(const FwdParams p) {
  constexpr int G = CELL == kGRU ? 3 : 4;
  constexpr int GD = G * DH;
  constexpr int NT = DH * 4;  // threads: 8 units x 4 gate slots per warp
  constexpr int WCH = GD / 4;  // 16-byte chunks of one Wx row
  static_assert(DH % 16 == 0, "four chains of whole float4s");
  __shared__ __align__(16) float hs[2][DH];
  __shared__ __align__(16) float xs[kPD][GD];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = p.T, B = p.B, NH = p.NH;
  const int head = blockIdx.x / B, b = blockIdx.x % B;
  const int g = lane & 3;                 // gate (GRU: slot 3 idle)
  const int j = warp * 8 + (lane >> 2);   // hidden unit
  const bool row_on = g < G;
  const int row = g * DH + j;             // gate row within the head
  const bool cell = g == 0;               // lane that applies the cell of unit j
  const float* Wx = static_cast<const float*>(p.Wx) + ((size_t)b * NH + head) * GD;
  const size_t wx_tstride = (size_t)B * NH * GD;
  const float* Rh = static_cast<const float*>(p.R) + (size_t)head * DH * GD;
  float* hseq = static_cast<float*>(p.h_seq) + ((size_t)b * NH + head) * DH + j;
  const size_t hseq_tstride = (size_t)B * NH * DH;
  const size_t si = ((size_t)b * NH + head) * DH + j;
  // element counts of the global buffers (bounds-check build)
  const long long n_state = (long long)B * NH * DH, n_hseq = (long long)T * n_state;
  const long long n_wx = (long long)T * B * NH * GD, n_r = (long long)NH * DH * GD;
  // (lanes without a gate row -- GRU slot 3 -- load nothing)
  const bool r_ok = !row_on || bc_ok((long long)head * DH * GD + (long long)(DH - 1) * GD + row, n_r, p.status);
  const bool s_ok = bc_ok((long long)si, n_state, p.status);

  unsigned long long rc2[DH / 2];  // (R[h][2i][row], R[h][2i + 1][row])
#pragma unroll
  for (int i = 0; i < DH / 2; ++i)
    rc2[i] = (row_on && r_ok)
                 ? pack2(Rh[(size_t)(2 * i) * GD + row], Rh[(size_t)(2 * i + 1) * GD + row])
                 : 0ull;
  const float brow =
      (row_on && p.bias && bc_ok((long long)head * GD + row, (long long)NH * GD, p.status))
          ? p.bias[(size_t)head * GD + row]
          : 0.f;

  float st_c = 0.f, st_n = 0.f, st_m = 0.f, st_h = 0.f;
  if (cell && s_ok) {
    st_h = p.h0 ? p.h0[si] : 0.f;
    st_c = p.c0 ? p.c0[si] : 0.f;
    st_n = p.n0 ? p.n0[si] : 0.f;
    st_m = p.m0 ? p.m0[si] : 0.f;
  }
  for (int i = tid; i < DH; i += NT)
    hs[0][i] = (p.h0 && bc_ok(((long long)b * NH + head) * DH + i, n_state, p.status))
                   ? p.h0[((size_t)b * NH + head) * DH + i]
                   : 0.f;

  auto issue = [&](int t) {
    if (t < T && tid < WCH &&
        bc_ok(((long long)b * NH + head) * GD + (long long)t * wx_tstride + 4 * tid + 3, n_wx, p.status))
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(&xs[t % kPD][4 * tid])),
                   "l"(Wx + (size_t)t * wx_tstride + 4 * tid)
                   : "memory");
    cp_async_commit();
  };
#pragma unroll 1
  for (int t = 0; t < kPD; ++t) issue(t);
  cp_async_wait<kPD - 1>();  // step 0 landed (own copies)
  __syncthreads();

#pragma unroll 1
  for (int t = 0; t < T; ++t) {
    // refill the slot of step t - 1 (read by every thread before the last
    // barrier) with step t - 1 + PD
    if (t > 0) issue(t - 1 + kPD);
    // 1. dot product over h_{t-1}: float4 i/4 feeds pair chains 2 ((i/4) % 2) + {0, 1}
    const float* hp = hs[t & 1];
    unsigned long long a2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int i = 0; i < DH; i += 4) {
      const float4 x = *reinterpret_cast<const float4*>(hp + i);
      const int c = 2 * ((i / 4) % 2);
      a2[c] = ffma2(pack2(x.x, x.y), rc2[i / 2], a2[c]);
      a2[c + 1] = ffma2(pack2(x.z, x.w), rc2[i / 2 + 1], a2[c + 1]);
    }
    const float rec = (((lo2(a2[0]) + hi2(a2[0])) + (lo2(a2[1]) + hi2(a2[1]))) +
                       ((lo2(a2[2]) + hi2(a2[2])) + (lo2(a2[3]) + hi2(a2[3])))) +
                      brow;  // R-part + bias of row `row`
    // 2. this lane's gate, then the unit's G values gathered into its cell lane
    const float* x = xs[t % kPD];
    const float xg = row_on ? x[row] : 0.f;
    const int base = lane & ~3;
    float v;
    if constexpr (CELL == kLSTM) {  // i, f, o: sigmoid; z: tanh
      const float th = tanhf(g == 2 ? rec + xg : 0.5f * (rec + xg));
      v = g == 2 ? th : fmaf(0.5f, th, 0.5f);
    } else if constexpr (CELL == kGRU) {  // r, z: sigmoid; n = tanh(x_n + r (R_n h + b_n))
      const float sg = fmaf(0.5f, tanhf(0.5f * (xg + rec)), 0.5f);
      const float r = __shfl_sync(0xffffffffu, sg, base);
      const float nt = tanhf(fmaf(r, rec, xg));
      v = g == 2 ? nt : sg;
    } else {  // sLSTM: i~, f~ raw (stabilised on the cell lane), z: tanh, o: sigmoid
      const float pre = rec + xg;
      const float th = tanhf(g == 3 ? 0.5f * pre : pre);
      v = g < 2 ? pre : (g == 2 ? th : fmaf(0.5f, th, 0.5f));
    }
    float gv[G];
#pragma unroll
    for (int k = 0; k < G; ++k) gv[k] = __shfl_sync(0xffffffffu, v, base + k);
    if (cell) {
      float h;
      if constexpr (CELL == kLSTM) {
        st_c = fmaf(gv[1], st_c, gv[0] * gv[2]);
        h = gv[3] * tanhf(st_c);
      } else if constexpr (CELL == kGRU) {
        h = (1.f - gv[1]) * gv[2] + gv[1] * st_h;
      } else {
        const float pi = gv[0], pf = gv[1];
        const float mn = fmaxf(pf + st_m, pi);
        const float ig = expf(pi - mn);
        const float fg = expf(pf + st_m - mn);
        st_c = fg * st_c + ig * gv[2];
        st_n = fg * st_n + ig;
        st_m = mn;
        h = gv[3] * (st_c / st_n);
      }
      st_h = h;
      hs[(t + 1) & 1][j] = h;
      if (bc_ok((long long)(hseq - static_cast<float*>(p.h_seq)), n_hseq, p.status)) *hseq = h;
    }
    hseq += hseq_tstride;
    // 3. step t + 1's Wx landed (own copies; PD - 2 younger groups may stay in
    //    flight); one barrier makes it and h_t visible to all
    cp_async_wait<kPD - 2>();
    __syncthreads();
  }
  cp_async_wait<0>();
  if (cell && T > 0) {
    if (!s_ok) return;
    if (p.hT) p.hT[si] = st_h;
    if (p.cT && CELL != kGRU) p.cT[si] = st_c;
    if (p.nT && CELL == kSLSTM) p.nT[si] = st_n;
    if (p.mT && CELL == kSLSTM) p.mT[si] = st_m;
  }
}

template <int CELL, int DH>
int launch_t(const FwdParams& p, cudaStream_t s, bool query_only, LaunchInfo* info) {
  constexpr int NT = DH * 4;
  const long long grid = (long long)p.NH * p.B;
  if (grid > 0x7fffffffLL) return (int)cudaErrorInvalidValue;
  if (info) *info = LaunchInfo{(int)grid, NT, 1, 1, 0, 1000 + CELL * 100 + DH};
  if (query_only) return 0;
  fwd_f32_kernel<CELL, DH><<<(int)grid, NT, 0, s>>>(p);
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
