// Persistent bf16 forward of the head-wise recurrence (LSTM / GRU / sLSTM).
//
// FlashRNN pages: the recurrent matrix stays on chip for the whole time loop
// (blog page, register-caching paragraph) and heads are independent blocks of
// a block-diagonal R mapped to separate thread blocks (blog page, head-wise
// paragraph).  On sm_103a one head (or one batch slice of a head) is one CTA;
// a head too large for one SM is split by hidden unit over the CTAs of a
// thread-block cluster, which exchange h_t through distributed shared memory.
//
// Per CTA: U = Dh / CS hidden units, all G gates of each unit.  Warp w owns UG
// units (G*UG gate rows = MT m16 tiles).  The contraction is "swap-AB":
//     acc[gate rows, batch] = R^T[gate rows, Dh] * h_{t-1}^T[Dh, batch]
// with R^T as the mma.sync A operand (fragments resident in registers; for
// very large heads the k-steps >= KREG sit in shared memory in fragment order)
// and h_{t-1} (bf16) as the B operand read by ldmatrix from a double buffer.
// Each compute warp streams its own Wx columns (G gates x UG units x 8 batch
// rows: one 16-byte cp.async per lane and step for UG = 8) PD steps ahead into
// a ring of PD stages, one cp.async group per step, so a step only waits on
// its own warp's copies (cp.async.wait_group) and no producer warp competes
// for an SM sub-partition's issue slots.  Each thread picks up its Wx values
// with one transposing ldmatrix, which lands them exactly in accumulator
// layout, and the accumulators start from Wx + bias.  Gate math runs on the accumulator
// registers; each thread owns whole (unit, batch) cells, so no gate exchange
// is needed.  Sigmoid gate rows of R, Wx and bias are pre-scaled by 1/2 so a
// sigmoid is one hardware tanh and one FMA: sigmoid(x) = (1 + tanh(x/2)) / 2.
//
// Exchange of h_t: CS == 1 -> shared memory + one named barrier per step.
// CS > 1 -> each warp stages its bf16 slice of h_t in shared memory, then its
// lanes send the slice's 16-byte chunks with st.async into every cluster CTA's
// buffer (lane -> one chunk, several ranks), completing bytes on that CTA's
// mbarrier; a CTA proceeds to step t+1 when all Dh*NB*2 bytes have landed.  Receiving all of h_t from a peer also
// proves the peer finished reading the buffer being overwritten next, so one
// double buffer suffices without a cluster barrier in the loop.
//
// Every wait is bounded (globaltimer); on expiry the kernel records
// kStatusTimeout in the status word, stops, lets in-flight copies land and
// exits through the same final barriers as a normal run.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "check.cuh"
#include "ptx.cuh"

namespace srnn {

template <int CELL, int DH, int UG, int NT, int KREG, int HS>
struct FwdCfg {
  static constexpr int G = CELL == kGRU ? 3 : 4;
  static constexpr int GD = G * DH;
  // m16 tiles per warp; GRU with 8 units per warp pads its 24 gate rows to 32
  static constexpr int MT = (UG * G + 15) / 16;
  static constexpr int ROWS = UG * G;     // gate rows that exist (the rest is padding)
  static constexpr int UGW = UG;          // hidden units per warp
  static constexpr int KS = DH / 16;      // k16 steps
  static constexpr int KSM = KS - KREG;   // k-steps whose A fragments live in smem
  static constexpr int NB = NT * 8;       // rows of the h buffer per CTA (n8 tiles)
  // HS = 1: h_{t-1} enters the MMA as a bf16 pair hi + lo (hi = bf16(h),
  // lo = bf16(h - hi)) in two B operands.  HS = 2: the pair shares one n8
  // tile -- rows 0-3 hold hi of four batch rows, rows 4-7 their lo -- so one
  // MMA covers both and the two column halves are summed by a lane shuffle.
  static constexpr int NBV = HS == 2 ? 4 : NB;  // batch rows per CTA
  static_assert(HS != 2 || NT == 1, "hi/lo n-tile pairing uses one n8 tile");
  // h row pitch in bytes: 16-byte chunks per row odd -> ldmatrix conflict-free
  static constexpr int HPB = ((DH * 2 / 16) % 2 == 0) ? DH * 2 + 16 : DH * 2;
  static constexpr int NSLOT = UG == 16 ? 2 : 1;  // units per thread
  static constexpr int NE = NSLOT * NT * 2;       // (unit, batch) cells per thread
  static constexpr int NTILE = G * NSLOT;         // 8x8 Wx tiles per thread and n-tile
  static constexpr int NQ = (NTILE + 3) / 4;      // ldmatrix instructions for them
  static constexpr int HPARTS = HS == 1 ? 2 : 1;  // h buffer parts
  // Wx prefetch depth in steps (ring stages): >= ~2 us of steps ahead
  static constexpr int PD = DH >= 256 ? 4 : 8;
  // long k chains run as two interleaved accumulator sets
  static constexpr bool SPLITK = KS >= 8 || HS;
  static_assert(KS >= 2, "two k16 steps at least");
  // cluster exchange: one warp's h_t slice (all parts) as 16-byte chunks
  static constexpr int STG_CH = HPARTS * NB * UG / 8;
  static constexpr int STG_BYTES = STG_CH * 16;
  static_assert(32 % STG_CH == 0, "staging chunks must tile a warp");
  // register estimate per compute thread -> largest CTA the register file holds
  static constexpr int REG_EST = MT * KREG * 4 + MT * NT * 8 + 88 + (HS == 1) * NT * 8;
  static constexpr int MAXT_R = (65536 / REG_EST) / 32 * 32;
  static constexpr int MAXT_0 = MAXT_R < 16 * 32 ? MAXT_R : 16 * 32;
  // The register file is split over the SM's four sub-partitions and warps are
  // spread over them, so a bound of 9 warps costs registers like 12 would; CTAs
  // come in 2^k warps (Dh 768: 3 x 2^k), so round to whole sub-partition rows.
  static constexpr int MAXT = MAXT_0 >= 256 ? MAXT_0 / 128 * 128 : MAXT_0;
  static_assert(UG == 8 || UG == 16, "unit group");
  static_assert(UG * G % 16 == 0 || (UG == 8 && G == 3), "gate rows per warp fill m16 tiles");
  static_assert(DH % 32 == 0, "Dh multiple of 32");
  static_assert(KREG >= 0 && KREG <= KS, "KREG");
  static_assert(NTILE % 2 == 0 || NTILE == 3, "Wx tiles come in pairs (or three: one x4 load)");
  // scale of gate g's preactivation: 1/2 for sigmoid gates on the fast path
  __host__ __device__ static constexpr float gate_scale(int g) {
    return HS ? 1.f
              : (CELL == kLSTM ? (g == 2 ? 1.f : 0.5f)
                               : (CELL == kGRU ? (g == 2 ? 1.f : 0.5f) : (g == 3 ? 0.5f : 1.f)));
  }
  // Wx row pitch in the ring (bytes): odd number of 16-byte chunks
  __host__ __device__ static constexpr uint32_t wx_pitch(int U) {
    return ((G * U * 2 / 16) % 2 == 0) ? G * U * 2 + 16 : G * U * 2;
  }
};

struct FwdSmem {
  uint32_t h, wx, rf, stg, bar, flag, total;
};

template <class C>
__host__ __device__ inline FwdSmem fwd_smem_layout(int U) {
  constexpr int NS = C::PD;
  FwdSmem L;
  const int NW = U / C::UGW;  // compute warps
  L.h = 0;
  uint32_t o = 2u * C::HPARTS * C::NB * C::HPB;
  o = (o + 127) & ~127u;
  L.wx = o;
  o += (uint32_t)NS * C::NB * C::wx_pitch(U);
  o = (o + 127) & ~127u;
  L.rf = o;
  o += (uint32_t)NW * C::MT * C::KSM * 512;
  o = (o + 15) & ~15u;
  L.stg = o;  // per warp: h_t staging for the cluster exchange, two parities
  o += (uint32_t)NW * C::STG_BYTES * 2;
  L.bar = o;
  o += 3 * 8;
  L.flag = o;
  o += 16;
  L.total = o;
  return L;
}

// Bounded wait on an mbarrier phase.  False: gave up (abort recorded).
template <bool CLUSTER_ACQ>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
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

// CL: the head is split over a thread-block cluster (CS > 1); TR: training stash.
template <int CELL, int DH, int UG, int NT, int KREG, int HS, int CL, int TR>
__global__ void __launch_bounds__(FwdCfg<CELL, DH, UG, NT, KREG, HS>::MAXT, 1)
    fwd_bf16_kernel(const FwdParams p) {
  using C = FwdCfg<CELL, DH, UG, NT, KREG, HS>;
  constexpr int G = C::G, GD = C::GD, MT = C::MT, KS = C::KS, KSM = C::KSM, NB = C::NB;
  constexpr int HPB = C::HPB, NE = C::NE, NSLOT = C::NSLOT, NTILE = C::NTILE, NQ = C::NQ;
  // Two k chains per m tile, and plain fp32 tanh: on GB300 tanh.approx.f16x2
  // takes 16 cycles of the multi-function unit per warp (two f32 tanh take the
  // same) and adds pack / unpack conversions (12 x 64 LSTM, one CTA per head:
  // 399 -> 383 ns per step with both changes).
  constexpr bool SPLITK = true;
  // HS = 1 (hi and lo as separate B operands) over >= 8 k16 steps: hi and lo
  // each on two chains (even/odd k pairs).  HS = 2: hi and lo in one n8 tile.
  constexpr bool HLO = HS == 1, HN = HS == 2;
  constexpr bool HS4 = HLO && KS >= 8;
  // A cluster step with >= 16 k16 steps: four k chains per m tile (k pair
  // parity x k16 half) -- the dependent mma.sync chain, not the issue rate,
  // bounds it (4x256 sLSTM: 8-long chains took ~640 cycles for 32 MMAs).
  // At 8 k16 steps two chains per tile measured faster.
  constexpr bool CH4 = !HLO && CL && KS >= 16;
  // One CTA per head (all warps meet at a barrier every step): the next step's
  // Wx is primed while this step's MMAs are in flight, in a second accumulator
  // set.  A cluster step primes it while h_t travels to the peers instead.
  constexpr bool EARLY_PREP = !CL && DH <= 128;
  extern __shared__ __align__(128) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int U = p.U, NW = U / UG, CS = p.CS, T = p.T, B = p.B, NH = p.NH;
  constexpr int PD = C::PD;
  const uint32_t crank = CL ? cluster_ctarank() : 0u;
  const int cid = blockIdx.x / CS;
  const int head = cid / p.nbslices, bslice = cid % p.nbslices;
  const int u0 = (int)crank * U;
  const int b0 = bslice * C::NBV;
  const int nvalid = min(C::NBV, B - b0);

  const FwdSmem L = fwd_smem_layout<C>(U);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t s_h = sbase + L.h, s_wx = sbase + L.wx, s_rf = sbase + L.rf;
  const uint32_t bar_h = sbase + L.bar;  // two: hfull[0], hfull[1]
  const uint32_t bar_dummy = bar_h + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.flag);
  const uint32_t WP = C::wx_pitch(U);
  const uint32_t stage_bytes = (uint32_t)NB * WP;
  const uint32_t hpart = 2u * NB * HPB;  // byte offset of the lo part of h
  const uint32_t htx = (uint32_t)C::HPARTS * NB * DH * 2;  // h bytes landing per step (cluster)
  // element counts of the global buffers (bounds-check build)
  const long long n_state = (long long)B * NH * DH, n_hseq = (long long)T * n_state;
  const long long n_wx = (long long)T * B * NH * GD, n_r = (long long)NH * DH * GD;
  const long long n_h_smem = 2ll * C::HPARTS * NB * HPB;  // h buffers (bytes from L.h)

  // ------------------------------------------------------------- set-up --
  if (tid == 0) {
    mbar_init(bar_h, 1);
    mbar_init(bar_h + 8, 1);
    mbar_init(bar_dummy, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // batch rows past B: their ring rows stay zero forever (never copied into)
  if (nvalid < NB) {
    const int per = (NB - nvalid) * (int)WP / 4;
    for (int i = tid; i < PD * per; i += blockDim.x) {
      const int s = i / per, r = i % per;
      *reinterpret_cast<uint32_t*>(smem + L.wx + s * stage_bytes + nvalid * WP + r * 4) = 0u;
    }
  }
  // h_{-1} = bf16(h0) for all Dh units of this batch slice into buffer 0
  // (HN: rows 4-7 take the residual parts of rows 0-3)
  for (int i = tid; i < NB * DH / 2; i += blockDim.x) {
    const int n = i / (DH / 2), j = 2 * (i % (DH / 2));
    const int nb = HN ? (n & 3) : n;
    float v0 = 0.f, v1 = 0.f;
    if (p.h0 != nullptr && nb < nvalid) {
      const long long e = ((long long)(b0 + nb) * NH + head) * DH + j;
      if (bc_ok(e + 1, n_state, p.status)) {
        v0 = p.h0[e];
        v1 = p.h0[e + 1];
      }
    }
    if (HN && n >= 4) {
      v0 -= bf16_round(v0);
      v1 -= bf16_round(v1);
    }
    if (!bc_ok((long long)n * HPB + j * 2 + 3, n_h_smem, p.status)) continue;
    *reinterpret_cast<uint32_t*>(smem + L.h + n * HPB + j * 2) = pack_bf16x2(v0, v1);
    if (HLO)
      *reinterpret_cast<uint32_t*>(smem + L.h + hpart + n * HPB + j * 2) =
          pack_bf16x2(v0 - bf16_round(v0), v1 - bf16_round(v1));
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (tid == 0 && CL) {
    // h_0 lands in buffer 1, h_1 in buffer 0 (first phase of each)
    if (T >= 2) mbar_arrive_expect_tx(bar_h + 8, htx);
    if (T >= 3) mbar_arrive_expect_tx(bar_h, htx);
  }
  if (CL) cluster_sync();
  else __syncthreads();

  const unsigned long long tlim = p.timeout_ns;

  {
    // ------------------------------------------------- compute warps --
    const uint16_t* Rb = static_cast<const uint16_t*>(p.R) + (size_t)head * DH * GD;
    const int ub = warp * UG;  // first CTA-local unit of this warp

    // A fragments of R^T: rows = (gate g, unit u) with row = g*UG + u; sigmoid
    // gate rows pre-scaled by 1/2 (exact in bf16).
    uint32_t areg[MT][KREG > 0 ? KREG : 1][4];
    const uint32_t rf_warp = s_rf + (uint32_t)warp * MT * KSM * 512 + lane * 16;
    auto rval = [&](int k, int col, float sc) -> uint32_t {
      if (col < 0) return 0u;
      if (!bc_ok((long long)head * DH * GD + (long long)k * GD + col, n_r, p.status)) return 0u;
      const uint16_t v = Rb[(size_t)k * GD + col];
      if (sc == 1.f) return v;
      const __nv_bfloat16 x = __float2bfloat16_rn(__uint_as_float((uint32_t)v << 16) * sc);
      return (uint32_t)(*reinterpret_cast<const uint16_t*>(&x));
    };
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int ra = mt * 16 + (lane >> 2), rb = ra + 8;
      const int ga = ra / UG, gb = rb / UG;
      // padding rows (GRU, 8 units per warp) get zero fragments
      const int ca = ra < C::ROWS ? ga * DH + u0 + ub + (ra % UG) : -1;
      const int cb = rb < C::ROWS ? gb * DH + u0 + ub + (rb % UG) : -1;
      const float sa = C::gate_scale(ga), sb = C::gate_scale(gb);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int k0 = ks * 16 + 2 * (lane & 3);
        uint32_t a[4];
        a[0] = rval(k0, ca, sa) | (rval(k0 + 1, ca, sa) << 16);
        a[1] = rval(k0, cb, sb) | (rval(k0 + 1, cb, sb) << 16);
        a[2] = rval(k0 + 8, ca, sa) | (rval(k0 + 9, ca, sa) << 16);
        a[3] = rval(k0 + 8, cb, sb) | (rval(k0 + 9, cb, sb) << 16);
        if (ks < KREG) {
#pragma unroll
          for (int q = 0; q < 4; ++q) areg[mt][ks < KREG ? ks : 0][q] = a[q];
        } else {
          const uint32_t addr = rf_warp + (uint32_t)(mt * KSM + (ks - KREG)) * 512;
          // the step loop reads the same offsets back
          if (!bc_ok((long long)(addr - s_rf) + 15, (long long)(L.stg > L.rf ? L.stg - L.rf : 0), p.status))
            continue;
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a[0]), "r"(a[1]),
                       "r"(a[2]), "r"(a[3])
                       : "memory");
        }
      }
    }

    // per-thread cells: slot us (unit lane/4 + 8us), n-tile nt, column e
    //   -> cell index (us*NT + nt)*2 + e, batch row nt*8 + 2*(lane&3) + e
    float sbias[G][NSLOT];  // gate_scale(g) * bias
#pragma unroll
    for (int us = 0; us < NSLOT; ++us) {
      const int j = u0 + ub + (lane >> 2) + 8 * us;
#pragma unroll
      for (int g = 0; g < G; ++g)
        sbias[g][us] = C::gate_scale(g) *
                       ((p.bias && bc_ok((long long)head * GD + g * DH + j, (long long)NH * GD, p.status))
                            ? p.bias[(size_t)head * GD + g * DH + j]
                            : 0.f);
      // HN: the lo columns (lanes with lane & 2) start from zero; the shuffle
      // adds them onto the hi columns, which carry Wx and the bias
      if (HN && (lane & 2)) {
#pragma unroll
        for (int g = 0; g < G; ++g) sbias[g][us] = 0.f;
      }
    }
    float st_c[NE], st_n[NE], st_m[NE], st_h[NE];
#pragma unroll
    for (int us = 0; us < NSLOT; ++us)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ei = (us * NT + nt) * 2 + e;
          // HN: a lo-column lane mirrors the state of its hi partner (lane ^ 2)
          const int n = (nt * 8 + 2 * (lane & 3) + e) & (HN ? 3 : 255);
          const int j = u0 + ub + (lane >> 2) + 8 * us;
          const size_t si = ((size_t)(b0 + n) * NH + head) * DH + j;
          const bool ok = n < nvalid && bc_ok((long long)si, n_state, p.status);
          st_c[ei] = (ok && p.c0) ? p.c0[si] : 0.f;
          st_n[ei] = (ok && p.n0) ? p.n0[si] : 0.f;
          st_m[ei] = (ok && p.m0) ? p.m0[si] : 0.f;
          st_h[ei] = (ok && p.h0) ? p.h0[si] : 0.f;
        }

    // ldmatrix (h, B operand): lane supplies row (lane & 7) of 8x8 matrix (lane >> 3)
    const uint32_t lm_off = (uint32_t)(lane & 7) * HPB + (uint32_t)(lane >> 3) * 16;
    // ldmatrix.trans (Wx): 8x8 tile k = us*G + g holds rows = batch, cols = the 8
    // units of slot us for gate g; the transpose hands lane l exactly the pair
    // (unit l/4, batch 2(l%4) and 2(l%4)+1) of its accumulator cells.
    uint32_t wx_off[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      int k = 4 * q + (lane >> 3);
      if (k >= NTILE) k -= 2;  // x2 form: lanes 16..31 supply ignored addresses
      const int us = k / G, g = k % G;
      wx_off[q] = (uint32_t)(lane & 7) * WP + (uint32_t)(g * U + ub + 8 * us) * 2;
    }
    // where this thread's cells go in the h buffers (batch row, unit)
    uint32_t h_off1[NSLOT][NT];
#pragma unroll
    for (int us = 0; us < NSLOT; ++us)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        h_off1[us][nt] = (uint32_t)(nt * 8 + 2 * (lane & 3)) * HPB +
                         (uint32_t)(u0 + ub + (lane >> 2) + 8 * us) * 2;
    // 16-byte rows of this warp's slice (UG units x NB rows): lane -> one row chunk,
    // used to ship h_t to the cluster peers and to store h_seq
    constexpr int NCH = NB * UG / 8;
    const int ch_n = lane / (UG / 8), ch_k = lane % (UG / 8);
    const bool ch_on = lane < NCH;
    const uint32_t ch_off = (uint32_t)ch_n * HPB + (uint32_t)(u0 + ub + 8 * ch_k) * 2;
    const bool ch_store = ch_on && ch_n < nvalid;
    __nv_bfloat16* hseq_ch = static_cast<__nv_bfloat16*>(p.h_seq) +
                             ((size_t)(ch_store ? b0 + ch_n : b0) * NH + head) * DH + u0 + ub + 8 * ch_k;
    const size_t hseq_tstride = (size_t)B * NH * DH;
    // cluster exchange: this warp's staging area [parity][part][row n][UG units];
    // lane -> chunk x_c = lane % STG_CH (part x_p, row x_n, 8 units at x_k), sent
    // to ranks lane / STG_CH, + 32 / STG_CH, ...
    constexpr int STG_CH = C::STG_CH, RSTEP = 32 / STG_CH;
    const uint32_t stg_warp = sbase + L.stg + (uint32_t)warp * C::STG_BYTES * 2;
    uint32_t stg_cell[NSLOT][NT];  // this thread's cells (e = 0) in the staging area
#pragma unroll
    for (int us = 0; us < NSLOT; ++us)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        stg_cell[us][nt] = (uint32_t)(nt * 8 + 2 * (lane & 3)) * (UG * 2) +
                           (uint32_t)((lane >> 2) + 8 * us) * 2;
    const int x_c = lane % STG_CH, x_r0 = lane / STG_CH;
    const int x_p = x_c / (NB * UG / 8), x_n = (x_c / (UG / 8)) % NB, x_k = x_c % (UG / 8);
    const uint32_t x_dst = (uint32_t)x_p * hpart + (uint32_t)x_n * HPB + (uint32_t)(u0 + ub + 8 * x_k) * 2;
    const bool x_store = x_r0 == 0 && x_p == 0 && x_n < nvalid;  // h_seq chunk owner
    __nv_bfloat16* hseq_x = static_cast<__nv_bfloat16*>(p.h_seq) +
                            ((size_t)(x_store ? b0 + x_n : b0) * NH + head) * DH + u0 + ub + 8 * x_k;
    bool dead = false;
    if (p.flags & (1 << 30)) {  // test hook: a barrier nothing ever completes
      if (!wait_phase<false>(bar_dummy, 0, abort_flag, p.status, tlim)) dead = true;
    }

    // this warp's Wx columns: G gates x UG units (UG/8 16-byte chunks) x nvalid
    // rows; lane -> chunks lane, lane + 32 (offsets fixed for all steps)
    constexpr int WCH = NB * G * (UG / 8), WCI = (WCH + 31) / 32;
    uint32_t wdst[WCI], wsrc[WCI];
    bool wok[WCI];
#pragma unroll
    for (int i = 0; i < WCI; ++i) {
      const int c = lane + 32 * i;
      const int n = c / (G * UG / 8), rem = c % (G * UG / 8), g = rem / (UG / 8), k = rem % (UG / 8);
      wok[i] = c < WCH && n < nvalid;
      wdst[i] = (uint32_t)n * WP + (uint32_t)(g * U + ub + 8 * k) * 2;
      wsrc[i] = (uint32_t)(n * NH * GD + g * DH + u0 + ub + 8 * k);
    }
    const __nv_bfloat16* wx_base =
        static_cast<const __nv_bfloat16*>(p.Wx) + ((size_t)b0 * NH + head) * GD;
    const size_t wx_tstride = (size_t)B * NH * GD;
    // copies of step tt into stage tt % PD, one commit group per step (empty past T)
    auto fetch = [&](int tt) {
      if (tt < T) {
        const uint32_t stage = s_wx + (uint32_t)(tt % PD) * stage_bytes;
        const __nv_bfloat16* src = wx_base + (size_t)tt * wx_tstride;
#pragma unroll
        for (int i = 0; i < WCI; ++i)
          if (wok[i] &&
              bc_ok(((long long)b0 * NH + head) * GD + (long long)tt * wx_tstride + wsrc[i] + 7, n_wx,
                    p.status) &&
              bc_ok((long long)(stage - s_wx) + wdst[i] + 15, (long long)PD * stage_bytes, p.status))
            cp_async16(stage + wdst[i], src + wsrc[i]);
      }
      cp_async_commit();
    };
#pragma unroll 1
    for (int tt = 0; tt < PD; ++tt) fetch(tt);
    int np = 0;  // steps primed so far (step np is next; its stage is np % PD)
    // accumulators of the step about to run, primed with scale*(Wx + bias)
    float acc[MT][NT][4], acc2[SPLITK ? MT : 1][NT][4];
    float acc3[HS4 || CH4 ? MT : 1][NT][4], acc4[HS4 || CH4 ? MT : 1][NT][4];
    float wxn[NE];  // GRU: Wx_n stays outside r*(R_n h + b_n)
    float accp[MT][NT][4], wxnp[NE];  // EARLY_PREP: primed for the next step
    float(*A)[NT][4] = EARLY_PREP ? accp : acc;
    float* WXN = EARLY_PREP ? wxnp : wxn;
    // Wait for the next Wx stage, move it into accumulator layout and release
    // the stage.  Runs while the step's MMAs are in flight (EARLY_PREP) or
    // after h_t is published, off the recurrence's critical path.
    uint32_t wxr[NT][NQ * 4];  // the next step's Wx values, raw bf16 pairs
    // First half of a prime: wait for step np's copies and load its values.
    // Cluster variants refill the stage the previous prime consumed (a whole
    // step ago) with step np - 1 + PD first, leaving PD - 1 younger groups in
    // flight.  The one-CTA variant (EARLY_PREP) runs this half at the top of a
    // step, before its MMAs (shared-memory instructions issued behind a burst of
    // mma.sync wait for the burst), and issues the refill later in the step
    // (late_fetch), so PD - 2 younger groups are in flight here.
    auto prep_load = [&]() {
      if (!EARLY_PREP) {
        if (np > 0) fetch(np - 1 + PD);
        cp_async_wait<PD - 1>();
      } else {
        if (np > 0) cp_async_wait<PD - 2>();
        else cp_async_wait<PD - 1>();
      }
      __syncwarp();
      const uint32_t stage = s_wx + (uint32_t)(np % PD) * stage_bytes;
      ++np;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const uint32_t addr = stage + nt * 8 * WP + wx_off[q];
          if (4 * q + 4 <= NTILE || NTILE - 4 * q == 3) {
            uint32_t r4[4];
            ldmatrix_x4_trans(r4, addr);
#pragma unroll
            for (int i = 0; i < 4; ++i) wxr[nt][4 * q + i] = r4[i];
          } else {
            uint32_t r2[2];
            ldmatrix_x2_trans(r2, addr);
            wxr[nt][4 * q] = r2[0];
            wxr[nt][4 * q + 1] = r2[1];
          }
        }
    };

    // The one-CTA refill of the stage step np - 2 used (this warp's own columns:
    // no other warp reads them) with step np - 2 + PD.  Issued after the gate
    // math, where the load/store unit is idle (at the top of a step it cost
    // ~35 ns more per step, 12 x 64 LSTM).
    auto late_fetch = [&]() {
      if (EARLY_PREP && np >= 2) fetch(np - 2 + PD);
    };
    // Second half: the loaded values into accumulator layout, scaled, plus bias.
    auto prep_fma = [&]() {
#pragma unroll
      for (int us = 0; us < NSLOT; ++us)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const uint32_t wv = wxr[nt][us * G + g];
              const float x = e ? bf16_hi(wv) : bf16_lo(wv);
              const int mt = UG == 16 ? g : g / 2;
              const int q = UG == 16 ? us * 2 + e : (g % 2) * 2 + e;
              if (CELL == kGRU && g == 2) {
                A[mt][nt][q] = sbias[g][us];
                WXN[(us * NT + nt) * 2 + e] = x;
              } else {
                A[mt][nt][q] = fmaf(C::gate_scale(g), x, sbias[g][us]);
              }
            }
      if (C::ROWS < MT * 16) {  // padding rows (GRU, 8 units per warp): start at zero
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) A[MT - 1][nt][2] = A[MT - 1][nt][3] = 0.f;
      }
    };
    auto prep = [&]() -> bool {
      prep_load();
      prep_fma();
      return true;
    };
    if (!dead && T > 0 && !prep()) dead = true;
    float hv[NE];  // h_t of this thread's cells (fp32)

    for (int t = 0; t < T; ++t) {
      // ---- wait for h_{t-1} (cluster)
      if (!dead && CL && t > 0) {
        if (!wait_phase<false>(bar_h + 8 * (t & 1), ((t - 1) >> 1) & 1, abort_flag, p.status, tlim))
          dead = true;
        else if (tid == 0 && t + 1 <= T - 2)
          mbar_arrive_expect_tx(bar_h + 8 * (t & 1), htx);  // for h_{t+1}
      }

      const bool send = t + 1 < T;
      if (!dead) {
        if (EARLY_PREP) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int q = 0; q < 4; ++q) acc[mt][nt][q] = accp[mt][nt][q];
          if (CELL == kGRU) {
#pragma unroll
            for (int ei = 0; ei < NE; ++ei) wxn[ei] = wxnp[ei];
          }
        }
        if (SPLITK) {
#pragma unroll
          for (int mt = 0; mt < (SPLITK ? MT : 1); ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int q = 0; q < 4; ++q) acc2[mt][nt][q] = 0.f;
        }
        if (HS4 || CH4) {
#pragma unroll
          for (int mt = 0; mt < (HS4 || CH4 ? MT : 1); ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int q = 0; q < 4; ++q) acc3[mt][nt][q] = acc4[mt][nt][q] = 0.f;
        }
        if (EARLY_PREP && send) prep_load();
        // ---- acc += R^T h_{t-1}
        const uint32_t hb = s_h + (uint32_t)(t & 1) * NB * HPB + lm_off;
        // (bounds-check build) the last 16 bytes this lane's ldmatrix reads; on
        // failure the step's contraction is skipped and the CTA stops
        const bool h_ok = bc_ok((long long)(hb - s_h) + (HLO ? hpart : 0) + (NT - 1) * 8 * HPB +
                                    (KS / 2 - 1) * 64 + 15,
                                n_h_smem, p.status);
        if (!h_ok) dead = true;
#pragma unroll
        for (int kp = 0; kp < (h_ok ? KS / 2 : 0); ++kp) {
          uint32_t bfr[NT][4], bfl[HLO ? NT : 1][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) ldmatrix_x4(bfr[nt], hb + nt * 8 * HPB + kp * 64);
          if (HLO) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              ldmatrix_x4(bfl[HLO ? nt : 0], hb + hpart + nt * 8 * HPB + kp * 64);
          }
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int ks = 2 * kp + hf;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              uint32_t a[4];
              if (ks < KREG) {
#pragma unroll
                for (int q = 0; q < 4; ++q) a[q] = areg[mt][ks < KREG ? ks : 0][q];
              } else {
                lds128(a, rf_warp + (uint32_t)(mt * KSM + (ks - KREG)) * 512);
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (HS4 && (kp & 1)) {  // odd k pairs: the second hi and lo chains
                  mma_bf16_16816(acc3[HS4 || CH4 ? mt : 0][nt], a, bfr[nt][2 * hf], bfr[nt][2 * hf + 1]);
                  mma_bf16_16816(acc4[HS4 || CH4 ? mt : 0][nt], a, bfl[HLO ? nt : 0][2 * hf],
                                 bfl[HLO ? nt : 0][2 * hf + 1]);
                } else if (CH4 && (kp & 1)) {  // odd k pairs: chains 3 and 4
                  mma_bf16_16816(hf ? acc4[HS4 || CH4 ? mt : 0][nt] : acc3[HS4 || CH4 ? mt : 0][nt], a,
                                 bfr[nt][2 * hf], bfr[nt][2 * hf + 1]);
                } else if (HLO) {  // hi and lo parts on two independent accumulator chains
                  mma_bf16_16816(acc[mt][nt], a, bfr[nt][2 * hf], bfr[nt][2 * hf + 1]);
                  mma_bf16_16816(acc2[SPLITK ? mt : 0][nt], a, bfl[HLO ? nt : 0][2 * hf],
                                 bfl[HLO ? nt : 0][2 * hf + 1]);
                } else if (SPLITK && hf == 1) {
                  mma_bf16_16816(acc2[SPLITK ? mt : 0][nt], a, bfr[nt][2], bfr[nt][3]);
                } else {
                  mma_bf16_16816(acc[mt][nt], a, bfr[nt][2 * hf], bfr[nt][2 * hf + 1]);
                }
              }
            }
          }
        }
        // next step's Wx into accumulator layout while the MMAs run
        if (EARLY_PREP && send) prep_fma();
        if (SPLITK) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if (HS4 || CH4)
                  acc[mt][nt][q] = (acc[mt][nt][q] + acc3[HS4 || CH4 ? mt : 0][nt][q]) +
                                   (acc2[mt][nt][q] + acc4[HS4 || CH4 ? mt : 0][nt][q]);
                else
                  acc[mt][nt][q] += acc2[SPLITK ? mt : 0][nt][q];
              }
        }
        if (HN) {  // hi column + lo column; both lanes of a pair get the same sum
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[mt][0][q] += __shfl_xor_sync(0xffffffffu, acc[mt][0][q], 2);
        }

        // ---- gate math and state update, one (unit, batch) cell at a time
        float act[TR ? 4 : 1][TR ? NE : 1];  // per-cell values the backward needs
#pragma unroll
        for (int us = 0; us < NSLOT; ++us)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int ei = (us * NT + nt) * 2 + e;
              float r[G];
#pragma unroll
              for (int g = 0; g < G; ++g)
                r[g] = UG == 16 ? acc[g][nt][us * 2 + e] : acc[g / 2][nt][(g % 2) * 2 + e];
              float h;
              if (CELL == kLSTM) {  // r[i,f,o] hold x/2
                const float2 t_if = make_float2(tanh_fast(r[0]), tanh_fast(r[1]));
                const float2 t_zo = make_float2(tanh_fast(r[2]), tanh_fast(r[3]));
                const float ig = fmaf(0.5f, t_if.x, 0.5f);
                const float fg = fmaf(0.5f, t_if.y, 0.5f);
                const float zg = t_zo.x;
                const float og = fmaf(0.5f, t_zo.y, 0.5f);
                const float c = fmaf(fg, st_c[ei], ig * zg);
                st_c[ei] = c;
                h = og * tanh_fast(c);
                if (TR) {
                  act[0][ei] = ig;
                  act[1][ei] = fg;
                  act[2][ei] = zg;
                  act[3][ei] = og;
                }
              } else if (CELL == kGRU) {  // r[r,z] hold x/2; r[n] = R_n h + b_n
                const float2 t_rz = make_float2(tanh_fast(r[0]), tanh_fast(r[1]));
                const float rg = fmaf(0.5f, t_rz.x, 0.5f);
                const float zg = fmaf(0.5f, t_rz.y, 0.5f);
                const float ng = tanh_fast(fmaf(rg, r[2], wxn[ei]));
                h = fmaf(zg, st_h[ei] - ng, ng);
                if (TR) {
                  act[0][TR ? ei : 0] = rg;
                  act[1][TR ? ei : 0] = zg;
                  act[2][TR ? ei : 0] = ng;
                  act[3][TR ? ei : 0] = r[2];  // R_n h + b_n
                }
              } else {
                const float pi = r[0], pf = r[1], pz = r[2], po = r[3];
                // m_t = max(f~ + m_{t-1}, i~): one of the two stabilised gates is
                // e^0 = 1, the other e^{-|f~ + m_{t-1} - i~|}
                const float fm = pf + st_m[ei];
                const bool fmax_ = fm >= pi;
                const float mn = fmax_ ? fm : pi;
                const float ex = __expf(-fabsf(fm - pi));
                const float ig = fmax_ ? ex : 1.f;
                const float fg = fmax_ ? 1.f : ex;
                // Exponentials from the ex2-based __expf (2 ulp).  HS: tanh z~ from
                // the identity tanh(x) = 1 - 2 / (e^{2x} + 1) on it -- the hardware
                // tanh.approx (~2^-11 relative) lets the exponential gating drift
                // 3e-2 from the exact recurrence over 4096 steps, this ~1e-6.
                const float zt = HS ? 1.f - __fdividef(2.f, __expf(2.f * pz) + 1.f) : tanh_fast(pz);
                const float c = fmaf(fg, st_c[ei], ig * zt);
                const float nn = fmaf(fg, st_n[ei], ig);
                st_c[ei] = c;
                st_n[ei] = nn;
                st_m[ei] = mn;
                // r[o] holds o~ (HS) or o~/2 (fast path).  HS: h = c / (n (1 + e^{-o~})),
                // one reciprocal for the output gate and the normaliser together.
                float og;
                if (HS) {
                  const float eo = 1.f + __expf(-po);
                  og = TR ? __fdividef(1.f, eo) : 0.f;
                  h = __fdividef(c, eo * nn);
                } else {
                  og = fmaf(0.5f, tanh_fast(po), 0.5f);
                  h = og * __fdividef(c, nn);
                }
                if (TR) {
                  act[0][TR ? ei : 0] = ig;
                  act[1][TR ? ei : 0] = fg;
                  act[2][TR ? ei : 0] = zt;
                  act[3][TR ? ei : 0] = og;
                }
              }
              hv[ei] = h;
              st_h[ei] = h;
            }

        late_fetch();
        // ---- publish h_t
        const uint32_t nbuf = s_h + (uint32_t)((t + 1) & 1) * NB * HPB;
        uint32_t xv[4] = {0u, 0u, 0u, 0u};  // cluster: this lane's 16-byte chunk of h_t
        if (CL) {
          // stage this warp's cells, then ship 16-byte chunks to every cluster CTA
          // (this one included) and store the h_seq chunk
          const uint32_t stg = stg_warp + (uint32_t)(t & 1) * C::STG_BYTES;
#pragma unroll
          for (int us = 0; us < NSLOT; ++us)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float hvv = hv[(us * NT + nt) * 2 + e];
                __nv_bfloat16 hi = __float2bfloat16_rn(hvv);
                if (HN && (lane & 2)) hi = __float2bfloat16_rn(hvv - __bfloat162float(hi));
                const uint32_t addr = stg + stg_cell[us][nt] + e * (UG * 2);
                asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr),
                             "h"(*reinterpret_cast<const uint16_t*>(&hi))
                             : "memory");
                if (HLO) {  // residual part: bf16(h - bf16(h))
                  const __nv_bfloat16 lo = __float2bfloat16_rn(hvv - __bfloat162float(hi));
                  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr + NB * UG * 2),
                               "h"(*reinterpret_cast<const uint16_t*>(&lo))
                               : "memory");
                }
              }
          __syncwarp();
          lds128(xv, stg + (uint32_t)x_c * 16);
          if (send) {
            const uint32_t lbar = bar_h + 8 * ((t + 1) & 1);
            const uint32_t ldst = nbuf + x_dst;
            if (bc_ok((long long)(ldst - s_h) + 15, n_h_smem, p.status))
              for (int rk = x_r0; rk < CS; rk += RSTEP) st_async_v4(mapa(ldst, rk), xv, mapa(lbar, rk));
          }
        } else {
          // own cells into the next buffer (also at the last step: h_seq is stored
          // from there after the barrier)
#pragma unroll
          for (int us = 0; us < NSLOT; ++us)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float hvv = hv[(us * NT + nt) * 2 + e];
                __nv_bfloat16 hi = __float2bfloat16_rn(hvv);
                if (HN && (lane & 2)) hi = __float2bfloat16_rn(hvv - __bfloat162float(hi));
                const uint32_t addr = nbuf + h_off1[us][nt] + e * HPB;
                asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr),
                             "h"(*reinterpret_cast<const uint16_t*>(&hi))
                             : "memory");
                if (HLO) {  // residual part: bf16(h - bf16(h))
                  const __nv_bfloat16 lo = __float2bfloat16_rn(hvv - __bfloat162float(hi));
                  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr + hpart),
                               "h"(*reinterpret_cast<const uint16_t*>(&lo))
                               : "memory");
                }
              }
        }
        // training stash of this step (after h_t is on its way: nothing of the
        // recurrence waits for it), per cell: four gate values [T,B,NH,4Dh] and
        // the state the backward needs [T,B,NH,Dh] (LSTM c_t, GRU h_t, sLSTM c_t
        // plus n_t in a third array).  GRU slots: r, z, n, R_n h + b_n.
        if (TR) {
#pragma unroll
          for (int us = 0; us < NSLOT; ++us)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int ei = (us * NT + nt) * 2 + e;
                const int n = nt * 8 + 2 * (lane & 3) + e;
                if (n < nvalid) {
                  const int j = u0 + ub + (lane >> 2) + 8 * us;
                  const size_t row = ((size_t)t * B + b0 + n) * NH + head;
                  if (!bc_ok((long long)(row * 4 * DH + 3 * DH + j), 4 * n_hseq, p.status) ||
                      !bc_ok((long long)(row * DH + j), n_hseq, p.status))
                    continue;
                  float* sg = p.stash_gates + row * 4 * DH + j;
#pragma unroll
                  for (int g = 0; g < 4; ++g) sg[g * DH] = act[TR ? g : 0][TR ? ei : 0];
                  p.stash_c[row * DH + j] = CELL == kGRU ? st_h[ei] : st_c[ei];
                  if (CELL == kSLSTM) p.stash_n[row * DH + j] = st_n[ei];
                }
              }
        }

        // ---- prime the next step's accumulators while other warps finish
        if (!EARLY_PREP && send && !prep()) dead = true;
        if (CL) {
          // this warp's h_seq chunk, after the exchange is on its way
          if (x_store &&
              bc_ok((long long)(hseq_x - static_cast<__nv_bfloat16*>(p.h_seq)) + 7, n_hseq, p.status))
            asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(hseq_x), "r"(xv[0]),
                         "r"(xv[1]), "r"(xv[2]), "r"(xv[3])
                         : "memory");
          hseq_x += hseq_tstride;
        }
      }
      if (!CL) {
        // h_t visible to every compute warp; a dead warp stops all of them together
        if (bar_red_or(1, NW * 32, dead)) break;
      } else if (dead) {
        break;
      }
      if (!CL) {
        // h_seq rows of this warp's slice after the barrier: they overlap the next step
        if (ch_store &&
            bc_ok((long long)(hseq_ch - static_cast<__nv_bfloat16*>(p.h_seq)) + 7, n_hseq, p.status)) {
          uint32_t v[4];
          lds128(v, s_h + (uint32_t)((t + 1) & 1) * NB * HPB + ch_off);
          asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(hseq_ch), "r"(v[0]), "r"(v[1]),
                       "r"(v[2]), "r"(v[3])
                       : "memory");
        }
        hseq_ch += hseq_tstride;
      }
    }
    if (!dead && T > 0) {  // final states (fp32)
#pragma unroll
      for (int us = 0; us < NSLOT; ++us)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int ei = (us * NT + nt) * 2 + e;
            const int n = nt * 8 + 2 * (lane & 3) + e;
            if (n >= nvalid) continue;
            const int j = u0 + ub + (lane >> 2) + 8 * us;
            const size_t si = ((size_t)(b0 + n) * NH + head) * DH + j;
            if (!bc_ok((long long)si, n_state, p.status)) continue;
            if (p.hT) p.hT[si] = hv[ei];
            if (p.cT && CELL != kGRU) p.cT[si] = st_c[ei];
            if (p.nT && CELL == kSLSTM) p.nT[si] = st_n[ei];
            if (p.mT && CELL == kSLSTM) p.mT[si] = st_m[ei];
          }
    }
    // let every issued Wx copy land before the CTA can exit
    cp_async_wait_all();
    __syncwarp();
  }
  // peers may still st.async into this CTA until they pass this point
  if (CL) cluster_sync();
}

template <int CELL, int DH, int UG, int NT, int KREG, int HS, int CL, int TR>
int launch_fwd_bf16_v(const FwdParams& p_in, cudaStream_t stream, bool query_only,
                      LaunchInfo* info) {
  using C = FwdCfg<CELL, DH, UG, NT, KREG, HS>;
  FwdParams p = p_in;
  auto kern = fwd_bf16_kernel<CELL, DH, UG, NT, KREG, HS, CL, TR>;
  const int NW = p.U / UG;
  const int threads = NW * 32;
  if (p.U % UG != 0 || NW < 1 || threads > C::MAXT) return (int)cudaErrorInvalidConfiguration;
  const uint32_t smem = fwd_smem_layout<C>(p.U).total;
  const int grid = p.NH * p.nbslices * p.CS;
  if (info) *info = LaunchInfo{grid, threads, p.CS, C::NBV, (int)smem, CELL * 100 + DH / 32 + 50 * HS};
  static int prepared[64][5];
  const int e = prepare_launch(prepared, kern, smem, threads, p.CS);
  if (e != 0) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.CS > 1 ? 1 : 0;
  if (query_only) return 0;
  return (int)cudaLaunchKernelEx(&cfg, kern, p);
}

// Launch limits of one compiled variant, for the host-side plan search: the
// largest CTA its register budget allows, its unit group and the dynamic
// shared memory a CTA of U units needs.
template <int CELL, int DH, int UG, int NT, int KREG, int HS = 0>
void fwd_bf16_limits_t(int U, FwdLimits* out) {
  using C = FwdCfg<CELL, DH, UG, NT, KREG, HS>;
  out->max_threads = C::MAXT;
  out->unit_group = UG;
  out->smem = (U > 0 && U % UG == 0) ? fwd_smem_layout<C>(U).total : 0u;
}

// Picks the cluster / training-stash variant of one (cell, Dh, unit group, KREG, HS).
// Heads that cannot fit one SM (Dh >= 256) only exist as cluster variants.
template <int CELL, int DH, int UG, int NT, int KREG, int HS = 0>
int launch_fwd_bf16_t(const FwdParams& p, cudaStream_t stream, bool query_only,
                      LaunchInfo* info) {
  const bool tr = (p.flags & 1) && p.stash_gates != nullptr;
  if (p.CS > 1) {
    if (tr) return launch_fwd_bf16_v<CELL, DH, UG, NT, KREG, HS, 1, 1>(p, stream, query_only, info);
    return launch_fwd_bf16_v<CELL, DH, UG, NT, KREG, HS, 1, 0>(p, stream, query_only, info);
  }
  if constexpr (DH <= 128) {
    if (tr) return launch_fwd_bf16_v<CELL, DH, UG, NT, KREG, HS, 0, 1>(p, stream, query_only, info);
    return launch_fwd_bf16_v<CELL, DH, UG, NT, KREG, HS, 0, 0>(p, stream, query_only, info);
  }
  return (int)cudaErrorInvalidConfiguration;
}

}  // namespace srnn
