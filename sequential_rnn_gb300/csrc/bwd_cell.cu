// Backward through time of the head-wise LSTM / GRU / sLSTM (bf16 operands,
// fp32 state).
//
// FlashRNN pages: the cells are trained (blog page, paragraph on gradient
// clipping and checkpointing during training); the recurrence runs in reverse
// with the same resident recurrent matrix.  For step t = T-1 .. 0 and every
// cell (b, j), from the values the training forward stashed:
//   LSTM  dh = dh_seq + dh_rec;  dc = dc' + dh*o*(1 - tanh(c)^2)
//         dG = [dc*z*i(1-i), dc*c_{t-1}*f(1-f), dc*i*(1-z^2), dh*tanh(c)*o(1-o)];  dc' <- dc*f
//   GRU   dh = dh_seq + dh_rec + dh'*z';  dn~ = dh(1-z)(1-n^2);  dz~ = dh(h_{t-1}-n)z(1-z)
//         dr~ = dn~*(R_n h + b_n)*r(1-r);  dWx = [dr~, dz~, dn~];  dG = [dr~, dz~, r*dn~]
//   sLSTM dh = dh_seq + dh_rec;  do = dh*c/n;  dc = dc' + dh*o/n;  dn = dn' - dh*o*c/n^2
//         dG = [(dc*z + dn)*i, (dc*c_{t-1} + dn*n_{t-1})*f, dc*i*(1-z^2), do*o(1-o)]
//         dc' <- dc*f, dn' <- dn*f   (the stabiliser m carries no gradient)
//   all   dh_rec[t-1] = dG_t @ R[h]^T;  dh0 = dh_rec[-1] (+ GRU direct term)
// dWx_t is written in the input dtype; db sums dG; dR = sum_t h_{t-1}^T dG_t is
// a GEMM afterwards (tc_gemm.cu).
//
// Layout on sm_103a: the CTAs of one thread-block cluster own disjoint hidden
// units of a head (U = Dh / CS each), as in the forward.  Per step a CTA forms
// dG for its own units, then computes on tensor cores the partial product of
// its own gate columns with R^T for ALL Dh units:
//     part[k, n] = sum_{own gate cols c} R[k, c] * dG[n, c]      (swap-AB mma.sync)
// and reduce-scatters it: bf16 partial rows of unit k go by st.async into the
// shared memory of the CTA owning k, which sums the CS partials in fp32.
// R's slice stays on chip for the whole loop (registers + shared memory).
// With CS == 1 the partial is already the full sum and stays local.
//
// Every wait is bounded; on expiry the kernel records a timeout in the status
// word and leaves through the same barriers as a normal run.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "check.cuh"
#include "ptx.cuh"

namespace srnn {
namespace {

constexpr int kNB = 8;  // batch rows per CTA (one mma n-tile)

// Per head size: cluster size, warps, k-steps of the R slice held in registers.
template <int DH>
struct BwdCfg;
template <> struct BwdCfg<32> { static constexpr int CS = 1, NW = 2, KREG = 8; };
template <> struct BwdCfg<64> { static constexpr int CS = 1, NW = 4, KREG = 16; };
template <> struct BwdCfg<128> { static constexpr int CS = 2, NW = 8, KREG = 16; };
template <> struct BwdCfg<256> { static constexpr int CS = 8, NW = 8, KREG = 8; };
template <> struct BwdCfg<768> { static constexpr int CS = 16, NW = 12, KREG = 4; };

template <int CELL, int DH>
struct BwdK {
  static constexpr int G = CELL == kGRU ? 3 : 4;
  static constexpr int CS = BwdCfg<DH>::CS, NW = BwdCfg<DH>::NW;
  static constexpr int U = DH / CS;            // units per CTA
  static constexpr int NTH = NW * 32;
  static constexpr int MTILES = DH / 16;       // m16 tiles over all units
  static constexpr int MTW = MTILES / NW;      // per warp
  static constexpr int KSW = G * U / 16;       // k16 steps over own gate columns
  static constexpr int KREG = BwdCfg<DH>::KREG < KSW ? BwdCfg<DH>::KREG : KSW;
  static constexpr int KSM = KSW - KREG;       // k-steps whose fragments sit in smem
  static constexpr int EPT = U * kNB / NTH;    // cells per thread
  // per-cell inputs of a step (stash values, previous states, upstream dh)
  static constexpr int NV = CELL == kLSTM ? 7 : (CELL == kGRU ? 6 : 9);
  static constexpr int DGP = ((G * U * 2 / 16) % 2 == 0) ? G * U * 2 + 16 : G * U * 2;  // dG row pitch
  static_assert(MTILES % NW == 0, "m tiles per warp");
  static_assert((U * kNB) % NTH == 0, "cells per thread");
  static_assert(U % 16 == 0, "own gate columns in whole k16 steps");
  // shared memory: [R frags][dG bf16 (B operand)][dh_rec exchange][barriers]
  static constexpr uint32_t RF = 0;
  static constexpr uint32_t RF_BYTES = (uint32_t)NW * MTW * KSM * 512;
  static constexpr uint32_t DG = (RF + RF_BYTES + 127) & ~127u;
  static constexpr uint32_t DG_BYTES = (uint32_t)kNB * DGP;
  static constexpr uint32_t RX = (DG + DG_BYTES + 127) & ~127u;
  // CS > 1: bf16 partials [2 buf][CS src][NB][U unit]; CS == 1: fp32 sums [NB][U]
  static constexpr uint32_t RX_BYTES = CS > 1 ? 2u * CS * U * kNB * 2 : (uint32_t)U * kNB * 4;
  // db scratch is used only after the last exchange: it aliases the dG and partial
  // buffers when they are large enough, else it gets its own region
  static constexpr uint32_t DB_BYTES = (uint32_t)kNB * G * U * 4;
  static constexpr bool DB_ALIAS = DB_BYTES <= RX + RX_BYTES - DG;
  static constexpr uint32_t DB = DB_ALIAS ? DG : ((RX + RX_BYTES + 127) & ~127u);
  static constexpr uint32_t BAR = ((DB_ALIAS ? RX + RX_BYTES : DB + DB_BYTES) + 15) & ~15u;
  static constexpr uint32_t FLAG = BAR + 16;
  // cluster reduce-scatter: per warp two 256-byte buffers, one m16 tile's
  // partials [batch row][16 units] bf16 each, sent as 16-byte chunks
  static constexpr uint32_t STG = (FLAG + 16 + 127) & ~127u;
  static constexpr uint32_t STG_BYTES = CS > 1 ? (uint32_t)NW * 2 * kNB * 16 * 2 : 0u;
  static constexpr uint32_t TOTAL = STG + STG_BYTES;
  static constexpr bool SPLIT = MTW <= 2;      // two k chains when registers allow
  // Per-cell inputs: loaded two steps ahead into registers where registers
  // allow (PFD = 2).  At Dh = 768 (168 registers) the allocator spills values
  // held across the MMA phase, and the spill store of a load in flight waits
  // out the whole memory latency; there (PFD = 0) the step's lines are
  // prefetched into L1 a step ahead and loaded while the step waits for dh_rec.
  static constexpr int PFD = DH >= 768 ? 0 : 2;
};

template <bool CLUSTER_ACQ>
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      int* status, unsigned long long limit_ns) {
  if (CLUSTER_ACQ ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (CLUSTER_ACQ ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

template <int CELL, int DH>
__global__ void __launch_bounds__(BwdK<CELL, DH>::NTH, 1) bwd_cell_kernel(const BwdParams p) {
  using K = BwdK<CELL, DH>;
  constexpr int G = K::G, CS = K::CS, U = K::U, MTW = K::MTW, KSW = K::KSW, KREG = K::KREG;
  constexpr int KSM = K::KSM, EPT = K::EPT, NTH = K::NTH, DGP = K::DGP, NV = K::NV;
  constexpr int GD = G * DH;
  constexpr bool CL = CS > 1;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T, B = p.B, NH = p.NH;
  const uint32_t crank = CL ? cluster_ctarank() : 0u;
  const int cid = blockIdx.x / CS;
  const int head = cid / p.nbslices, bslice = cid % p.nbslices;
  const int u0 = (int)crank * U;
  const int b0 = bslice * kNB;
  const int nvalid = min(kNB, B - b0);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t s_rf = sbase + K::RF, s_dg = sbase + K::DG, s_rx = sbase + K::RX;
  const uint32_t s_stg = sbase + K::STG + (uint32_t)warp * (2 * kNB * 16 * 2);
  const uint32_t bar_r = sbase + K::BAR;  // two: partial buffers 0 / 1
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + K::FLAG);
  const unsigned long long tlim = p.timeout_ns;
  constexpr uint32_t kTx = (uint32_t)CS * U * kNB * 2;  // partial bytes landing per step
  // element counts of the global buffers (bounds-check build)
  const long long n_state = (long long)B * NH * DH, n_seq = (long long)T * n_state;
  const long long n_g = (long long)T * B * NH * GD, n_r = (long long)NH * DH * GD;

  if (tid == 0) {
    mbar_init(bar_r, 1);
    mbar_init(bar_r + 8, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // partials of step s (s = T-1-t, s = 0..T-1) land in buffer s&1 with phase s>>1
  if (CL && tid == 0) {
    mbar_arrive_expect_tx(bar_r, kTx);
    if (T >= 2) mbar_arrive_expect_tx(bar_r + 8, kTx);
  }
  if (CL) cluster_sync();

  // ---- A fragments: rows = all Dh units k (warp's m tiles), cols = own gate
  //      columns c = g*U + u  ->  R[k][g*Dh + u0 + u]
  const uint16_t* Rb = static_cast<const uint16_t*>(p.R) + (size_t)head * DH * GD;
  uint32_t areg[MTW][KREG > 0 ? KREG : 1][4];
  const uint32_t rf_warp = s_rf + (uint32_t)warp * MTW * KSM * 512 + lane * 16;
#pragma unroll
  for (int mt = 0; mt < MTW; ++mt) {
    const int ra = (warp * MTW + mt) * 16 + (lane >> 2), rb = ra + 8;
#pragma unroll
    for (int ks = 0; ks < KSW; ++ks) {
      const int c0 = ks * 16 + 2 * (lane & 3);
      auto col = [&](int c) { return (c / U) * DH + u0 + (c % U); };
      auto rv = [&](int r, int c) -> uint32_t {
        const long long e = (long long)r * GD + col(c);
        return bc_ok((long long)head * DH * GD + e, n_r, p.status) ? (uint32_t)Rb[e] : 0u;
      };
      uint32_t a[4];
      a[0] = rv(ra, c0) | (rv(ra, c0 + 1) << 16);
      a[1] = rv(rb, c0) | (rv(rb, c0 + 1) << 16);
      a[2] = rv(ra, c0 + 8) | (rv(ra, c0 + 9) << 16);
      a[3] = rv(rb, c0 + 8) | (rv(rb, c0 + 9) << 16);
      if (ks < KREG) {
#pragma unroll
        for (int q = 0; q < 4; ++q) areg[mt][ks < KREG ? ks : 0][q] = a[q];
      } else if (bc_ok((long long)(rf_warp - s_rf) + (mt * KSM + (ks - KREG)) * 512 + 15, K::RF_BYTES,
                       p.status)) {  // the step loop reads the same offsets back
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                         rf_warp + (uint32_t)(mt * KSM + (ks - KREG)) * 512),
                     "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3])
                     : "memory");
      }
    }
  }

  // ---- cells: ci = tid + e*NTH -> batch row n = ci / U, own unit u = ci % U
  int cu[EPT], cn[EPT];
  bool cok[EPT];
  // carries: LSTM dc; GRU dh*z (direct path to h_{t-1}); sLSTM dc and dn
  float dcar[EPT], dncar[EPT], dbacc[EPT][G], dhv[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int ci = tid + e * NTH;
    cu[e] = ci % U;
    cn[e] = ci / U;
    const size_t si = ((size_t)(b0 + cn[e]) * NH + head) * DH + u0 + cu[e];
    cok[e] = cn[e] < nvalid && bc_ok((long long)si, n_state, p.status);
    dcar[e] = (CELL != kGRU && cok[e] && p.dcT) ? p.dcT[si] : 0.f;
    dncar[e] = (CELL == kSLSTM && cok[e] && p.dnT) ? p.dnT[si] : 0.f;
    dhv[e] = (cok[e] && p.dhT) ? p.dhT[si] : 0.f;  // dh_rec of the last step
#pragma unroll
    for (int g = 0; g < G; ++g) dbacc[e][g] = 0.f;
  }
  const __nv_bfloat16* dhs = static_cast<const __nv_bfloat16*>(p.dh_seq);
  __nv_bfloat16* dwx = static_cast<__nv_bfloat16*>(p.dWx);
  __nv_bfloat16* drec = static_cast<__nv_bfloat16*>(p.drec);
  const size_t tstep = (size_t)B * NH;  // rows per time step
  // per-step inputs of one cell (see NV): the stash row of step t, the state of
  // step t-1 (or the initial state), and the upstream dh
  auto load_step = [&](int t, int e, float (&v)[NV]) {
    if (t < 0 || !cok[e]) {
#pragma unroll
      for (int q = 0; q < NV; ++q) v[q] = 0.f;
      return;
    }
    const size_t row = ((size_t)t * B + b0 + cn[e]) * NH + head;
    const int j = u0 + cu[e];
    const size_t si0 = ((size_t)(b0 + cn[e]) * NH + head) * DH + j;  // initial-state index
    if (!bc_ok((long long)(row * 4 * DH + 3 * DH + j), 4 * n_seq, p.status) ||
        !bc_ok((long long)(row * DH + j), n_seq, p.status) ||
        !(t > 0 ? bc_ok((long long)((row - tstep) * DH + j), n_seq, p.status)
               : bc_ok((long long)si0, n_state, p.status))) {
#pragma unroll
      for (int q = 0; q < NV; ++q) v[q] = 0.f;
      return;
    }
    const float* sg = p.stash_gates + row * 4 * DH + j;
#pragma unroll
    for (int g = 0; g < 4; ++g) v[g] = sg[g * DH];
    if (CELL == kLSTM) {
      v[4] = p.stash_c[row * DH + j];
      v[5] = t > 0 ? p.stash_c[(row - tstep) * DH + j] : (p.c_init ? p.c_init[si0] : 0.f);
    } else if (CELL == kGRU) {
      v[4] = t > 0 ? p.stash_c[(row - tstep) * DH + j] : (p.h_init ? p.h_init[si0] : 0.f);
    } else {
      v[4] = p.stash_c[row * DH + j];
      v[5] = p.stash_n[row * DH + j];
      v[6] = t > 0 ? p.stash_c[(row - tstep) * DH + j] : (p.c_init ? p.c_init[si0] : 0.f);
      v[7] = t > 0 ? p.stash_n[(row - tstep) * DH + j] : (p.n_init ? p.n_init[si0] : 0.f);
    }
    v[NV - 1] = __bfloat162float(dhs[row * DH + j]);
  };
  constexpr int PFD = K::PFD;
  // the same cell's input lines, into L1 only
  auto prefetch_step = [&](int t, int e) {
    if (t < 0 || !cok[e]) return;
    const size_t row = ((size_t)t * B + b0 + cn[e]) * NH + head;
    const int j = u0 + cu[e];
    if (!bc_ok((long long)(row * 4 * DH + 3 * DH + j), 4 * n_seq, p.status) ||
        !bc_ok((long long)(row * DH + j), n_seq, p.status))
      return;
    const float* sg = p.stash_gates + row * 4 * DH + j;
#pragma unroll
    for (int g = 0; g < 4; ++g) prefetch_l1(sg + g * DH);
    prefetch_l1(p.stash_c + row * DH + j);
    if (t > 0) prefetch_l1(p.stash_c + (row - tstep) * DH + j);
    if (CELL == kSLSTM) {
      prefetch_l1(p.stash_n + row * DH + j);
      if (t > 0) prefetch_l1(p.stash_n + (row - tstep) * DH + j);
    }
    prefetch_l1(dhs + row * DH + j);
  };
  float bufA[EPT][NV], bufB[PFD == 2 ? EPT : 1][NV];  // inputs of steps t (A) and t-1 (B)
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    if (PFD == 2) {
      load_step(T - 1, e, bufA[e]);
      load_step(T - 2, e, bufB[PFD == 2 ? e : 0]);
    } else {
      prefetch_step(T - 1, e);
    }
  }

  // B operand (dG) ldmatrix address of this lane
  const uint32_t lm_off = (uint32_t)(lane & 7) * DGP + (uint32_t)(lane >> 3) * 16;
  bool dead = false;

  // one reverse step s (t = T-1-s) on the inputs in `cur`; refills `cur` with the
  // inputs of step t-2 (two buffers alternate: the loads get two steps to land),
  // or (PFD = 0) loads them at the start of the step from L1.
  // Returns true when the loop ends (s == T yields dh0, or every thread gave up).
  auto rstep = [&](int s, float (&cur)[EPT][NV]) -> bool {
    const int t = T - 1 - s;
    if (PFD == 0 && s < T) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) load_step(t, e, cur[e]);
    }
    // ---- dh_rec[t] from the partials of step s-1
    if (s > 0) {
      if (CL) {
        const int ps = s - 1;
        if (!dead && !bwait<false>(bar_r + 8 * (ps & 1), (ps >> 1) & 1, abort_flag, p.status, tlim))
          dead = true;
        if (!dead) {
          if (tid == 0 && ps + 2 <= T - 1) mbar_arrive_expect_tx(bar_r + 8 * (ps & 1), kTx);
          const uint8_t* rx = smem + K::RX + (ps & 1) * (CS * U * kNB * 2);
#pragma unroll
          for (int e = 0; e < EPT; ++e) {
            float acc = 0.f;
#pragma unroll
            for (int src = 0; src < CS; ++src)
              acc += bf16_to_f32(*reinterpret_cast<const uint16_t*>(
                  rx + ((src * kNB + cn[e]) * U + cu[e]) * 2));
            dhv[e] = acc;
          }
        }
      } else {
        const float* rx = reinterpret_cast<const float*>(smem + K::RX);
#pragma unroll
        for (int e = 0; e < EPT; ++e) dhv[e] = rx[cn[e] * U + cu[e]];
      }
    }
    if (s == T) return true;  // dh_rec[-1] is in dhv

    // ---- pointwise backward of this step's cells -> dG (bf16 to smem), dWx
    if (!dead) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        const float* v = cur[e];
        float dg[G], dx[G];  // recurrent-preactivation gradient, input-projection gradient
        if (CELL == kLSTM) {
          const float ig = v[0], fg = v[1], zg = v[2], og = v[3], c = v[4], cp = v[5];
          const float dh = v[6] + dhv[e];
          const float tc = tanhf(c);
          const float dc = fmaf(dh * og, 1.f - tc * tc, dcar[e]);
          dg[0] = dc * zg * ig * (1.f - ig);
          dg[1] = dc * cp * fg * (1.f - fg);
          dg[2] = dc * ig * (1.f - zg * zg);
          dg[3] = dh * tc * og * (1.f - og);
          dcar[e] = dc * fg;
#pragma unroll
          for (int g = 0; g < G; ++g) dx[g] = dg[g];
        } else if (CELL == kGRU) {
          const float rg = v[0], zg = v[1], ng = v[2], rn = v[3], hp = v[4];
          const float dh = v[5] + dhv[e] + dcar[e];
          const float dnp = dh * (1.f - zg) * (1.f - ng * ng);
          const float dzp = dh * (hp - ng) * zg * (1.f - zg);
          const float drp = dnp * rn * rg * (1.f - rg);
          dx[0] = dg[0] = drp;
          dx[1] = dg[1] = dzp;
          dx[2] = dnp;
          dg[2] = dnp * rg;
          dcar[e] = dh * zg;
        } else {
          const float ig = v[0], fg = v[1], zg = v[2], og = v[3];
          const float c = v[4], nn = v[5], cp = v[6], np = v[7];
          const float dh = v[8] + dhv[e];
          const float rn = 1.f / nn;
          const float dc = fmaf(dh * og, rn, dcar[e]);
          const float dn = dncar[e] - dh * og * c * rn * rn;
          dg[0] = fmaf(dc, zg, dn) * ig;
          dg[1] = fmaf(dc, cp, dn * np) * fg;
          dg[2] = dc * ig * (1.f - zg * zg);
          dg[3] = dh * c * rn * og * (1.f - og);
          dcar[e] = dc * fg;
          dncar[e] = dn * fg;
#pragma unroll
          for (int g = 0; g < G; ++g) dx[g] = dg[g];
        }
        const size_t row = ((size_t)t * B + b0 + cn[e]) * NH + head;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const __nv_bfloat16 vg = __float2bfloat16_rn(dg[g]);
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(s_dg + cn[e] * DGP + (g * U + cu[e]) * 2),
                       "h"(*reinterpret_cast<const uint16_t*>(&vg))
                       : "memory");
          if (cok[e] && bc_ok((long long)(row * GD + g * DH + u0 + cu[e]), n_g, p.status)) {
            dwx[row * GD + g * DH + u0 + cu[e]] = __float2bfloat16_rn(dx[g]);
            if (CELL == kGRU && drec) drec[row * GD + g * DH + u0 + cu[e]] = vg;
          }
          dbacc[e][g] += cok[e] ? dg[g] : 0.f;
        }
      }
      // inputs of step t-2 arrive while the exchange runs
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        if (PFD == 2) load_step(t - 2, e, cur[e]);
        else prefetch_step(t - 1, e);
      }
    }
    // dG of all cells in shared memory (and the previous dh_rec fully read)
    if (bar_red_or(1, NTH, dead)) return true;

    // ---- partial[k, n] = sum_{own cols} R[k, c] dG[n, c] for this warp's k tiles
    constexpr bool SPLIT = K::SPLIT;
    float acc[MTW][4], acc2[SPLIT ? MTW : 1][4];
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[mt][q] = acc2[SPLIT ? mt : 0][q] = 0.f;
#pragma unroll
    for (int kp = 0; kp < (KSW + 1) / 2; ++kp) {
      uint32_t bfr[4];
      if (2 * kp + 1 < KSW) {
        ldmatrix_x4(bfr, s_dg + lm_off + kp * 64);
      } else {  // odd tail: one k16 step (lanes 16..31 supply unused addresses)
        uint32_t b2[2];
        asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                     : "=r"(b2[0]), "=r"(b2[1])
                     : "r"(s_dg + (uint32_t)(lane & 7) * DGP + (uint32_t)((lane >> 3) & 1) * 16 + kp * 64));
        bfr[0] = b2[0];
        bfr[1] = b2[1];
        bfr[2] = bfr[3] = 0u;
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int ks = 2 * kp + hf;
        if (ks >= KSW) continue;
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt) {
          uint32_t a[4];
          if (ks < KREG) {
#pragma unroll
            for (int q = 0; q < 4; ++q) a[q] = areg[mt][ks < KREG ? ks : 0][q];
          } else {
            lds128(a, rf_warp + (uint32_t)(mt * KSM + (ks - KREG)) * 512);
          }
          if (SPLIT && hf) mma_bf16_16816(acc2[SPLIT ? mt : 0], a, bfr[2], bfr[3]);
          else mma_bf16_16816(acc[mt], a, bfr[2 * hf], bfr[2 * hf + 1]);
        }
      }
    }
    // ---- reduce-scatter: rows k (unit) go to the CTA owning k.  Cluster: a
    // tile's 16 units x 8 batch rows are staged as bf16 in one of the warp's two
    // buffers and leave as 16 chunks of 8 units (16 bytes), one st.async.v4 per
    // lane of the first half-warp (four-byte words per lane were 4x the remote
    // stores); a tile of 16 units never straddles two owners (U % 16 == 0).
    // Rows 4-7 keep their two 16-byte halves swapped, so the staging writes of
    // rows n and n + 4 (32 bytes apart x 4) fall on different banks.
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt) {
      const int n = 2 * (lane & 3);
      const int kt = (warp * MTW + mt) * 16;  // first unit of this tile
      const uint32_t stg = s_stg + (uint32_t)(mt & 1) * (kNB * 16 * 2);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int k = kt + (lane >> 2) + 8 * half;
        const float v0 = acc[mt][2 * half] + (SPLIT ? acc2[SPLIT ? mt : 0][2 * half] : 0.f);
        const float v1 =
            acc[mt][2 * half + 1] + (SPLIT ? acc2[SPLIT ? mt : 0][2 * half + 1] : 0.f);
        // pair units (k, k+1) of one batch row with the neighbour lane (k^1): the
        // even lane keeps batch n, the odd one batch n+1; rows stay unit-contiguous
        const bool kev = ((lane >> 2) & 1) == 0;
        const float other = __shfl_xor_sync(0xffffffffu, kev ? v1 : v0, 4);
        const float p0 = kev ? v0 : other, p1 = kev ? other : v1;
        const int nn = n + (kev ? 0 : 1), ke = k & ~1;
        if (CL) {
          const int kl = ke - kt, ch = (kl >> 3) ^ ((nn >> 2) & 1);  // physical 16-byte half
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(stg + (uint32_t)(nn * 32 + ch * 16 + (kl & 7) * 2)),
                       "r"(pack_bf16x2(p0, p1))
                       : "memory");
        } else {
          *reinterpret_cast<float2*>(smem + K::RX + (nn * U + ke) * 4) = make_float2(p0, p1);
        }
      }
      if (CL) {
        __syncwarp();  // the tile is staged (and the buffer's previous chunks were read)
        if (lane < 16) {
          const int cn = lane >> 1, k0 = kt + 8 * (lane & 1);
          uint32_t v[4];
          lds128(v, stg + (uint32_t)(cn * 32 + (((lane & 1) ^ ((cn >> 2) & 1)) * 16)));
          const int owner = k0 / U, ku = k0 % U;
          const uint32_t buf = (uint32_t)(s & 1) * (CS * U * kNB * 2);
          const uint32_t laddr = s_rx + buf + (uint32_t)((crank * kNB + cn) * U + ku) * 2;
          if (bc_ok((long long)(laddr - s_rx) + 15, K::RX_BYTES, p.status) && bc_ok(owner, CS, p.status))
            st_async_v4(mapa(laddr, owner), v, mapa(bar_r + 8 * (s & 1), owner));
        }
      }
    }
    if (!CL) {
      // partials complete; also orders the next step's dG writes after these reads
      if (bar_red_or(1, NTH, dead)) return true;
    }
    return false;
  };
  for (int s = 0;; s += 2) {
    if (rstep(s, bufA)) break;
    if constexpr (PFD == 2) {
      if (rstep(s + 1, bufB)) break;
    } else {
      if (rstep(s + 1, bufA)) break;
    }
  }

  // ---- initial-state gradients and this slice's bias-gradient partial (every
  //      exchange is done: the last pass consumed the final partials, so the
  //      buffers can be reused)
  if (!dead) {
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      if (!cok[e]) continue;
      const size_t si = ((size_t)(b0 + cn[e]) * NH + head) * DH + u0 + cu[e];
      if (!bc_ok((long long)si, n_state, p.status)) continue;
      if (p.dh0) p.dh0[si] = dhv[e] + (CELL == kGRU ? dcar[e] : 0.f);
      if (p.dc0 && CELL != kGRU) p.dc0[si] = dcar[e];
      if (p.dn0 && CELL == kSLSTM) p.dn0[si] = dncar[e];
    }
  }
  __syncthreads();
  float* dbs = reinterpret_cast<float*>(smem + K::DB);  // [n][g][u]
#pragma unroll
  for (int e = 0; e < EPT; ++e)
#pragma unroll
    for (int g = 0; g < G; ++g) dbs[(cn[e] * G + g) * U + cu[e]] = dbacc[e][g];
  __syncthreads();
  if (p.db_part && !dead) {
    for (int i = tid; i < G * U; i += NTH) {
      const int g = i / U, u = i % U;
      float sum = 0.f;
      for (int n = 0; n < kNB; ++n) sum += dbs[(n * G + g) * U + u];
      if (bc_ok(((long long)bslice * NH + head) * GD + g * DH + u0 + u, (long long)p.nbslices * NH * GD,
                p.status))
        p.db_part[((size_t)bslice * NH + head) * GD + g * DH + u0 + u] = sum;
    }
  }
  if (CL) cluster_sync();
}

template <int CELL, int DH>
int launch_t(const BwdParams& p_in, cudaStream_t s, bool query_only, LaunchInfo* info) {
  using K = BwdK<CELL, DH>;
  BwdParams p = p_in;
  p.CS = K::CS;
  p.U = K::U;
  auto kern = bwd_cell_kernel<CELL, DH>;
  const int grid = p.NH * p.nbslices * K::CS;
  if (info) *info = LaunchInfo{grid, K::NTH, K::CS, kNB, (int)K::TOTAL, 500 + CELL * 100 + DH / 32};
  static int prepared[64][5];
  const int e = prepare_launch(prepared, kern, K::TOTAL, K::NTH, K::CS);
  if (e != 0) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(K::NTH);
  cfg.dynamicSmemBytes = K::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = K::CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = K::CS > 1 ? 1 : 0;
  if (query_only) return 0;
  return (int)cudaLaunchKernelEx(&cfg, kern, p);
}

template <int CELL>
int launch_cell(const BwdParams& p, int Dh, cudaStream_t s, bool q, LaunchInfo* info) {
  switch (Dh) {
    case 32: return launch_t<CELL, 32>(p, s, q, info);
    case 64: return launch_t<CELL, 64>(p, s, q, info);
    case 128: return launch_t<CELL, 128>(p, s, q, info);
    case 256: return launch_t<CELL, 256>(p, s, q, info);
    case 768: return launch_t<CELL, 768>(p, s, q, info);
    default: return (int)cudaErrorInvalidValue;
  }
}

}  // namespace

int launch_bwd_bf16(const BwdParams& p, int cell, int Dh, cudaStream_t s, bool query_only,
                    LaunchInfo* info) {
  if (cell == kLSTM) return launch_cell<kLSTM>(p, Dh, s, query_only, info);
  if (cell == kGRU) return launch_cell<kGRU>(p, Dh, s, query_only, info);
  return launch_cell<kSLSTM>(p, Dh, s, query_only, info);
}

}  // namespace srnn
