// Input projection Wx = x W^T + b on CTA pairs: tcgen05.mma.cta_group::2.
//
// A cluster of two CTAs (two SMs) computes one 256 x 256 output tile.  Each
// CTA stages its own half of the operands -- rows m0 + 128 r .. + 127 of x and
// rows n0 + 128 r .. + 127 of W (r = the CTA's rank in the pair) -- and the
// MMA, issued by one thread of the even CTA, reads both halves: the pair's
// tensor cores share the B operand, so each SM brings in 32 KB of operands per
// 64-deep k block instead of the 48 KB a one-SM 128 x 256 tile needs (64 B per
// clock at the tensor rate instead of 96).  Each CTA's TMEM holds the fp32
// accumulator of its 128 rows x 256 columns, double-buffered (512 columns), so
// a tile's epilogue overlaps the next tile's MMAs.
//
//   warp 0    TMA producer (one lane; both CTAs, each its own half; the bytes
//             complete on the even CTA's stage barrier) and TMEM owner,
//   warp 1    MMA issuer (one lane of the even CTA): 4 pair MMAs per k block,
//             then a commit that frees the stage in both CTAs, and one per tile
//             that hands both accumulators to the epilogues,
//   warps 2-9 epilogue, two per 32-lane TMEM quarter (warp w reads lanes
//             32 (w % 4) ..), each 128 of the 256 columns: tcgen05.ld, bf16
//             (+ bias) through shared memory and TMA stores; each warp then
//             arrives on the even CTA's accumulator-empty barrier (16 arrivals
//             per tile).  Eight warps, not four: with four the drain of a tile
//             took longer than its MMAs (~10k cycles against ~6k per tile).
//
// Two pairs per cluster (four SMs) for deep sums (K >= 2048) when N spans two
// 256-column blocks: the pairs take neighbouring column blocks of the same 256
// rows, so they stage the same x rows; CTA r of each pair fetches half of
// those 128 rows and multicasts them into CTA r of both pairs (their bytes
// complete on each destination pair's even-CTA barrier), and every stage is
// released only when both pairs' MMAs have read it.  x then crosses from L2
// once per two tiles: 24 KB instead of 32 KB of operands per SM and k block.
//
// Every wait is bounded; a wait that runs out sets the status word and stops
// the CTA's loops, and the teardown lets every copy and commit that targets a
// CTA land before any CTA of the cluster exits.
//
// FlashRNN pages: the input projection is ordinary dense work outside the
// sequential part (blog page, register-caching paragraph).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "tc.cuh"
#include "tc_epi.cuh"

namespace srnn {
namespace {

constexpr int PBM = 256, PBN = 256, PBK = 64;  // pair tile (128 rows per CTA), k block
constexpr int PNSTG = 6;                      // ring stages
constexpr uint32_t P_TILE = 128 * PBK * 2;    // 16 KB: this CTA's half of A (or of B)
constexpr uint32_t P_STAGE = 2 * P_TILE;      // 32 KB
constexpr int P_NEPI = 8;                     // epilogue warps
constexpr int P_THREADS = 32 * (2 + P_NEPI);
constexpr uint32_t P_OUT = P_NEPI * 4096;     // epilogue staging, 4 KB per warp
constexpr uint32_t P_BIAS = P_NEPI * 128;     // epilogue bias slots, 128 B per warp
constexpr uint32_t P_TMEM_COLS = 2 * PBN;     // two accumulator buffers
// ring + staging + bias + 1024 for aligning them + barriers (full, empty,
// tfull x2, tempty x2) + TMEM slot and flags (no static shared memory: its
// padding would not leave room)
constexpr uint32_t P_SMEM = PNSTG * P_STAGE + P_OUT + P_BIAS + 1024 + (2 * PNSTG + 4) * 8 + 16;

struct PairArgs {
  int M, N;             // output rows / columns
  int tiles_m, tiles_n; // 256-row blocks, column groups (256 columns per pair of the cluster)
  int full;             // units run whole: unit u by cluster u % clusters
  int halves;           // the other units, split in two along N: half h by cluster h
  int nkb;              // 64-deep k blocks
  const float* bias;    // [N] or null
  int* status;
  unsigned long long timeout_ns;
};

// mbarrier wait bounded by `limit_ns`; a timeout sets the abort flag and the
// status word.  The barriers order tensor-core and TMA work (async proxy) and
// tcgen05 accesses bracketed by tcgen05 fences; no generic-proxy data crosses
// the pair through them, so the CTA-scope acquire of a plain try_wait serves
// (the cluster-scope form cost ~80 cycles per 64-deep k block on the MMA
// thread's critical path).
__device__ __forceinline__ bool wait_pair(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// A cluster's i-th work unit: 256 rows from m0; pair p of the cluster takes the
// nw columns (256, or 128 for a half unit) from n0 + p * nw.
struct PairUnit {
  int m0, n0, nw;
};
// Cluster c runs units c, c + clusters, ... below g.full, then half c if
// c < g.halves: the last wave's units are split so that no cluster runs a
// whole extra one.
__device__ __forceinline__ int pair_units(const PairArgs& g, int c, int ncl) {
  return (c < g.full ? (g.full - c + ncl - 1) / ncl : 0) + (c < g.halves ? 1 : 0);
}
template <int NP>
__device__ __forceinline__ PairUnit pair_unit(const PairArgs& g, int c, int ncl, int i) {
  const int u = c + i * ncl;
  PairUnit w;
  if (u < g.full) {
    w.m0 = (u / g.tiles_n) * PBM;
    w.n0 = (u % g.tiles_n) * NP * PBN;
    w.nw = PBN;
  } else {
    const int t = g.full + c / 2;
    w.m0 = (t / g.tiles_n) * PBM;
    w.n0 = (t % g.tiles_n) * NP * PBN + (c & 1) * NP * (PBN / 2);
    w.nw = PBN / 2;
  }
  return w;
}

// NP pairs per cluster.  NP = 2: the two pairs share their 256 rows of x (they
// take neighbouring column blocks), and each x half-tile is fetched once from
// L2: CTA r of pair p loads rows 64 p .. 64 p + 63 of the 128 rows both CTAs
// r of the cluster stage, multicast to both.
template <int NP>
__global__ void __launch_bounds__(P_THREADS, 1)
    tc_proj_pair_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB,
                        const __grid_constant__ CUtensorMap mC, const PairArgs g) {
  static_assert(NP == 1 || NP == 2, "one or two pairs per cluster");
  constexpr int CS = 2 * NP;                               // CTAs per cluster
  constexpr uint16_t kAll = (uint16_t)((1u << CS) - 1u);   // every CTA of the cluster
  extern __shared__ __align__(16) uint8_t smem_raw[];
  // Every CTA runs this layout from the same shared-window base, so an offset
  // names the same buffer in any CTA (the pair MMA and the multicast rely on it).
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;  // 128-byte swizzle: 1024-byte aligned tiles
  const uint32_t out_stage = ring + PNSTG * P_STAGE;
  const uint32_t bias_s = out_stage + P_OUT;
  const uint32_t bar_full = bias_s + P_BIAS, bar_empty = bar_full + 8 * PNSTG;
  const uint32_t bar_tfull = bar_empty + 8 * PNSTG, bar_tempty = bar_tfull + 16;
  const uint32_t tslot = bar_tempty + 16;
  // flags after the TMEM slot: abort, copies issued, copies consumed
  int* const flags = reinterpret_cast<int*>(smem_raw + (tslot + 4 - raw));
  volatile int* abort_flag = flags;
  int& issued_s = flags[1];
  int& consumed_s = flags[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t r = rank & 1u;              // 0: the CTA of its pair that issues the MMAs
  const uint32_t pp = rank >> 1;             // pair of the cluster
  const uint32_t lead = rank & ~1u;          // this pair's even CTA
  const uint16_t pair_mask = (uint16_t)(0x3u << lead);
  const int cl = blockIdx.x / CS, ncl = gridDim.x / CS;
  const int nunits = pair_units(g, cl, ncl);
  const unsigned long long tlim = g.timeout_ns;

  if (threadIdx.x == 32) {
    for (int s = 0; s < PNSTG; ++s) {
      mbar_init(bar_full + 8 * s, 1);    // the even CTA's expect_tx arrival (+ the pair's bytes)
      mbar_init(bar_empty + 8 * s, NP);  // one commit per pair: every pair writes this stage
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);   // the pair commit
      mbar_init(bar_tempty + 8 * a, 2 * P_NEPI);  // the epilogue warps of both CTAs of the pair
    }
    flags[0] = 0;
    issued_s = 0;
    consumed_s = 0;
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc_pair(tslot, P_TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every CTA's barriers exist before any copy or arrival targets them
  tc_fence_after();
  uint32_t tmem;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(tslot) : "memory");
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      tma_prefetch_map(&mA);
      tma_prefetch_map(&mB);
      const uint32_t lead_full = mapa(bar_full, lead);
      int it = 0;  // ring position across all units
      bool stop = false;
      for (int i = 0; i < nunits && !stop; ++i) {
        const PairUnit w = pair_unit<NP>(g, cl, ncl, i);
        // a half unit's pair MMA reads the first 64 of each CTA's 128 staged W rows
        const int ma = w.m0 + (int)r * 128, nb = w.n0 + (int)pp * w.nw + (int)r * (w.nw / 2);
        for (int kb = 0; kb < g.nkb; ++kb, ++it) {
          const int s = it % PNSTG, ph = it / PNSTG;
          // every pair's MMAs on this stage's previous contents completed
          if (it >= PNSTG && !wait_pair(bar_empty + 8 * s, (ph - 1) & 1, abort_flag, g.status, tlim)) {
            stop = true;
            break;
          }
          const uint32_t sA = ring + s * P_STAGE, sB = sA + P_TILE;
          // the even CTA's barrier counts the bytes landing in both CTAs of its
          // pair; the other CTAs' copies may land before this arrival (the
          // transaction count goes below zero until then, and the phase cannot
          // complete without the arrival)
          if (r == 0) mbar_arrive_expect_tx(bar_full + 8 * s, 2 * P_STAGE);
          if (NP == 1) {
            tma_load_2d_pair(sA, &mA, kb * PBK, ma, lead_full + 8 * s);
          } else {
            // rows 64 pp .. + 63 of the x half-tile, into CTA r of both pairs
            tma_load_2d_pair_mc(sA + pp * (P_TILE / 2), &mA, kb * PBK, ma + (int)pp * 64,
                                lead_full + 8 * s, (uint16_t)((1u << r) | (1u << (r + 2))));
          }
          tma_load_2d_pair(sB, &mB, kb * PBK, nb, lead_full + 8 * s);
        }
      }
      issued_s = it;
      // every commit aimed at this CTA's stage barriers has arrived before the
      // CTA may leave (the last PNSTG stages' commits are not waited on above)
      if (!stop) {
        for (int k = it - PNSTG < 0 ? 0 : it - PNSTG; k < it; ++k)
          if (!wait_pair(bar_empty + 8 * (k % PNSTG), (k / PNSTG) & 1, abort_flag, g.status, tlim))
            break;
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0 && r == 0) {
      constexpr uint32_t idesc_full = idesc_bf16_f32(PBM, PBN, false, false);
      constexpr uint32_t idesc_half = idesc_bf16_f32(PBM, PBN / 2, false, false);
      int it = 0;
      bool stop = false;
      for (int i = 0; i < nunits && !stop; ++i) {
        const uint32_t idesc = pair_unit<NP>(g, cl, ncl, i).nw == PBN ? idesc_full : idesc_half;
        const int a = i & 1;
        // both CTAs' epilogues have drained this accumulator buffer (unit i - 2)
        if (i >= 2 && !wait_pair(bar_tempty + 8 * a, ((i >> 1) - 1) & 1, abort_flag, g.status, tlim))
          break;
        tc_fence_after();
        const uint32_t dacc = tmem + (uint32_t)(a * PBN);
        for (int kb = 0; kb < g.nkb; ++kb, ++it) {
          const int s = it % PNSTG, ph = it / PNSTG;
          if (!wait_pair(bar_full + 8 * s, ph & 1, abort_flag, g.status, tlim)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t sA = ring + s * P_STAGE, sB = sA + P_TILE;
#pragma unroll
          for (int k4 = 0; k4 < PBK / 16; ++k4) {
            // K step of 16: 32 bytes along the K-major rows of both halves
            const uint64_t ad = sdesc_sw128(sA + k4 * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sB + k4 * 32, 16, 1024);
            umma_bf16_pair(dacc, ad, bd, idesc, (kb != 0 || k4 != 0) ? 1u : 0u);
          }
          umma_commit_pair(bar_empty + 8 * s, kAll);  // stage reusable by every pair's copies
        }
        if (!stop) umma_commit_pair(bar_tfull + 8 * a, pair_mask);  // unit done -> both epilogues
      }
      consumed_s = it;
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int hc = (warp - 2) >> 2;   // column half of the tile
    const int e = warp - 2;           // staging buffer / bias slot
    const uint32_t lead_tempty = mapa(bar_tempty, lead);
    for (int i = 0; i < nunits; ++i) {
      const int a = i & 1;
      if (!wait_pair(bar_tfull + 8 * a, (i >> 1) & 1, abort_flag, g.status, tlim)) break;
      tc_fence_after();
      const PairUnit w = pair_unit<NP>(g, cl, ncl, i);
      if (w.nw == PBN || hc == 0)  // a half unit's 128 columns: the first four warps
        epilogue_bf16_bias_128(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * PBN + hc * 128),
                               g.bias, w.n0 + (int)pp * w.nw + hc * 128, g.N,
                               w.m0 + (int)r * 128 + q * 32, g.M, out_stage + (uint32_t)e * 4096,
                               bias_s + (uint32_t)e * 128, &mC);
      // accumulator buffer a may be overwritten by unit i + 2
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (r == 0) mbar_arrive(bar_tempty + 8 * a);
        else mbar_arrive_remote(lead_tempty + 8 * a);
      }
    }
    if (lane == 0) bulk_wait_read_all();  // the output stores have left shared memory
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every CTA done issuing copies, MMAs and arrivals
  if (r == 0 && warp == 0 && lane == 0) {
    // After a timeout: let every copy any CTA of the cluster issued land (the
    // bytes landing in this pair complete on this CTA's stage barriers) before
    // the cluster may exit.
    int hi = issued_s;
    for (int k = 0; k < CS; ++k) {
      int other = 0;
      asm volatile("ld.shared::cluster.u32 %0, [%1];"
                   : "=r"(other)
                   : "r"(mapa(tslot + 8, (uint32_t)k))
                   : "memory");
      hi = other > hi ? other : hi;
    }
    if (*abort_flag || consumed_s < hi) {
      for (int k = consumed_s; k < hi; ++k) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar_full + 8 * (k % PNSTG), (k / PNSTG) & 1))
          if (globaltimer_ns() - t0 > 10000000ull) break;
      }
    }
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, P_TMEM_COLS);
  }
}

}  // namespace

// bf16 row-major map helper of tc_gemm.cu
int make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t pitch,
             uint32_t bx, uint32_t by);

namespace {

// Clusters of `cs` CTAs of `kern` that can be resident at once (0: none).
template <class Kern>
int active_clusters(int (&cache)[64], Kern kern, int cs) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev] != 0) return cache[dev] > 0 ? cache[dev] : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cs);
  cfg.blockDim = dim3(P_THREADS);
  cfg.dynamicSmemBytes = P_SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  if (dev >= 0 && dev < 64) cache[dev] = n > 0 ? n : -1;
  return n;
}

// One launch with NP pairs per cluster; -1 when no such cluster can run here
// (NP = 2: also when such clusters would leave more than 8 SMs idle).
template <int NP>
int launch_pair_np(const void* x, const void* W, const float* bias, void* Wx, int M, int N, int K,
                   int* status, unsigned long long timeout_ns, cudaStream_t s, int max_ctas) {
  constexpr int CS = 2 * NP;
  auto kern = tc_proj_pair_kernel<NP>;
  static int prepared[64][5];
  static int active[64];
  const int e = prepare_launch(prepared, kern, P_SMEM, P_THREADS, CS);
  if (e != 0) return e;
  PairArgs g{};
  g.M = M;
  g.N = N;
  g.tiles_m = (M + PBM - 1) / PBM;
  g.tiles_n = (N + NP * PBN - 1) / (NP * PBN);
  g.nkb = (K + PBK - 1) / PBK;
  g.bias = bias;
  g.status = status;
  g.timeout_ns = timeout_ns;
  const long long units = (long long)g.tiles_m * g.tiles_n;
  if (units > 0x3fffffffLL) return (int)cudaErrorInvalidValue;
  if (units == 0) return 0;
  int cap = sm_count();
  if (max_ctas > 0 && max_ctas < cap) cap = max_ctas;
  long long ncl = cap / CS;
  // (after prepare_launch: the occupancy query needs the kernel's shared-memory opt-in)
  const int act = active_clusters(active, kern, CS);
  if (NP == 2 && CS * act < sm_count() - 8) return -1;
  if (act < ncl) ncl = act;
  if (units < ncl) ncl = units;
  if (ncl < 1) return -1;
  // the last wave's r units as 2r halves when they fit one wave (768 pair tiles
  // over 76 pairs: 8 pairs would run an 11th whole tile, 16 run half of one)
  const long long rem = units % ncl;
  const bool split = rem > 0 && 2 * rem <= ncl;
  g.full = (int)(split ? units - rem : units);
  g.halves = (int)(split ? 2 * rem : 0);
  CUtensorMap a, b, c;
  // NP = 2: each CTA fetches half of its 128 x rows (the other half arrives by
  // the other pair's multicast)
  int r = make_map(&a, x, (uint64_t)M, (uint64_t)K, (uint64_t)K, 64, NP == 2 ? 64 : 128);
  if (r) return r;
  r = make_map(&b, W, (uint64_t)N, (uint64_t)K, (uint64_t)K, 64, 128);
  if (r) return r;
  r = make_map(&c, Wx, (uint64_t)M, (uint64_t)N, (uint64_t)N, 64, 32);  // output boxes
  if (r) return r;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(CS * ncl));
  cfg.blockDim = dim3(P_THREADS);
  cfg.dynamicSmemBytes = P_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, kern, a, b, c, g);
}

}  // namespace

// Wx [M, N] = x [M, K] W[N, K]^T + bias on CTA pairs: two pairs per cluster
// sharing x for deep sums (K >= 2048) when such clusters cover all but a few
// SMs and the columns fill both pairs, else one pair per cluster.  Measured on
// GB300, where 36 four-CTA clusters (144 of 152 SMs) fit: 16384 x 3072 x 3072
// 168.6 against 173.3 us; at K = 768 the idle SMs and a longer last wave cost
// more than the shared x saves (54.0 against 52.8 us).  Returns -1 when no
// pair can be co-scheduled or fewer than two CTAs are allowed (the caller then
// takes the one-CTA kernel), 0 on success, else a CUDA error code.
int launch_input_proj_pair(const void* x, const void* W, const float* bias, void* Wx, int M, int N,
                           int K, int* status, unsigned long long timeout_ns, cudaStream_t s,
                           int max_ctas) {
  if (N >= 2 * PBN && K >= 2048 && (max_ctas <= 0 || max_ctas >= sm_count())) {
    const int e = launch_pair_np<2>(x, W, bias, Wx, M, N, K, status, timeout_ns, s, max_ctas);
    if (e != -1) return e;
  }
  return launch_pair_np<1>(x, W, bias, Wx, M, N, K, status, timeout_ns, s, max_ctas);
}

}  // namespace srnn
