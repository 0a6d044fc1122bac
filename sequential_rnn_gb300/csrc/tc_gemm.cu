// Dense bf16 GEMMs of the path on the 5th-generation tensor cores:
//
//   dR[h] = sum_{t,b} h_{t-1}[b,h,:]^T dG_t[b,h,:]          (weight gradient)
//   Wx    = x W^T + b                                       (input projection)
//
// Persistent kernel, one CTA per SM, looping over work units (head z, 128-row
// tile, BN-column tile, K split).  A unit's fp32 128 x BN tile accumulates in
// tensor memory by tcgen05.mma (M=128, N=BN, K=16 per instruction) from
// 128-byte-swizzled shared-memory tiles that TMA loads through a ring:
//   warp 0   TMA producer (one lane) and TMEM owner (alloc / dealloc),
//   warp 1   MMA issuer (one lane): 4 MMAs per 64-deep k block, then a
//            tcgen05.commit that frees the ring stage once they completed,
//            and one per unit that hands the accumulator to the epilogue,
//   warps 2-5 epilogue: tcgen05.ld of their 32-lane TMEM quarter (one output
//            row per thread), then fp32 (stored, or added for K splits) or
//            bf16(+bias) stores.
// The accumulator is double-buffered in TMEM (2 x BN columns), so a unit's
// epilogue overlaps the next unit's MMAs, and the ring keeps streaming
// across units.
// Operands may be K-major (rows of K) or MN-major (rows of M / N, as both
// operands of dR are: K = (t, b) is the row index of h_seq and of dG).
// The K range is one or two segments, each with its own tensor maps and row
// offsets: dR takes k in [0, B) from h0 and the rest from h_seq, against dG
// rows [0, B) and [B, T*B).  K tails and rows past a tensor's end read zeros.
//
// FlashRNN pages: the recurrent weight R is the only part that must stay
// sequential (blog page, register-caching paragraph); everything else is
// ordinary dense work, here on the tensor cores.
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

constexpr int TBM = 128, TBK = 64;

enum : int { kOutF32 = 0, kOutBf16Bias = 1, kOutF32Add = 2 };

template <int BN, int OUT>
struct TcCfg {
  static constexpr uint32_t TILE_A = TBM * TBK * 2;        // 16 KB
  static constexpr uint32_t TILE_B = BN * TBK * 2;         // 16 or 32 KB
  static constexpr uint32_t STAGE = TILE_A + TILE_B;
  static constexpr int NSTG = BN == 256 ? 4 : 6;
  static constexpr uint32_t TMEM_COLS = 2 * BN;            // two accumulator buffers
  // bf16 output: per epilogue warp two 32-row x 64-column boxes staged for TMA stores
  static constexpr uint32_t OUT_STAGE = OUT == kOutBf16Bias ? 4 * 8192 : 0;
  // bf16 output: per epilogue warp a 32-value bias slot (the 32 columns it converts)
  static constexpr uint32_t BIAS = OUT == kOutBf16Bias ? 4 * 32 * 4 : 0;
  // ring + output staging + bias + 1024 for aligning them + barriers (full,
  // empty, tfull x2, tempty x2) + TMEM slot
  static constexpr uint32_t SMEM = NSTG * STAGE + OUT_STAGE + BIAS + 1024 + (2 * NSTG + 4) * 8 + 16;
};

struct GemmArgs {
  int M, N;                // valid output rows / columns per batch item z
  int Z, tiles_m, tiles_n, ksplit;
  int m_off_z, n_off_z;    // A's M and B's N coordinate offset per z (head)
  int nkb0, nkb1;          // 64-deep k blocks in segment 0 and 1
  int ka0[2], kb0[2];      // K coordinate offsets of A and B per segment
  void* C;                 // output [z][M][ldc]
  long long c_stride_z;
  int ldc;
  const float* bias;       // [N] (kOutBf16Bias; may be null)
  int* status;
  unsigned long long timeout_ns;
};

struct Unit {
  int z, m_base, n_base, kb_lo, kb_hi;
};

__device__ __forceinline__ Unit unit_of(const GemmArgs& g, int u) {
  Unit w;
  const int ks = u % g.ksplit;
  int r = u / g.ksplit;
  const int nt = r % g.tiles_n;
  r /= g.tiles_n;
  const int mt = r % g.tiles_m;
  w.z = r / g.tiles_m;
  w.m_base = mt * TBM;
  w.n_base = nt;  // scaled by BN by the caller
  const int nkb = g.nkb0 + g.nkb1;
  w.kb_lo = (int)((long long)nkb * ks / g.ksplit);
  w.kb_hi = (int)((long long)nkb * (ks + 1) / g.ksplit);
  return w;
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
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

template <bool A_MN, bool B_MN, int OUT, int BN>
__global__ void __launch_bounds__(192, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mB0,
                   const __grid_constant__ CUtensorMap mA1, const __grid_constant__ CUtensorMap mB1,
                   const __grid_constant__ CUtensorMap mC, const GemmArgs g) {
  using C = TcCfg<BN, OUT>;
  constexpr int NSTG = C::NSTG;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ int abort_flag_s;
  __shared__ int issued_s, consumed_s;
  volatile int* abort_flag = &abort_flag_s;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;  // 128-byte swizzle: 1024-byte aligned tiles
  const uint32_t out_stage = ring + NSTG * C::STAGE;  // 1024-byte aligned
  const uint32_t bias_s = out_stage + C::OUT_STAGE;
  const uint32_t bar_full = bias_s + C::BIAS, bar_empty = bar_full + 8 * NSTG;
  const uint32_t bar_tfull = bar_empty + 8 * NSTG, bar_tempty = bar_tfull + 16;
  const uint32_t tslot = bar_tempty + 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nunits = g.Z * g.tiles_m * g.tiles_n * g.ksplit;

  if (threadIdx.x == 32) {
    for (int s = 0; s < NSTG; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 4);  // one arrival per epilogue warp
    }
    abort_flag_s = 0;
    issued_s = 0;
    consumed_s = 0;
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(tslot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t tmem;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(tslot) : "memory");
  const unsigned long long tlim = g.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      tma_prefetch_map(&mA0);
      tma_prefetch_map(&mB0);
      if (g.nkb1) {
        tma_prefetch_map(&mA1);
        tma_prefetch_map(&mB1);
      }
      int it = 0;  // ring position across all units
      bool stop = false;
      for (int u = blockIdx.x; u < nunits && !stop; u += gridDim.x) {
        const Unit w = unit_of(g, u);
        const int mA = w.m_base + w.z * g.m_off_z, nB = w.n_base * BN + w.z * g.n_off_z;
        for (int kb = w.kb_lo; kb < w.kb_hi; ++kb, ++it) {
          const int s = it % NSTG, ph = it / NSTG;
          if (it >= NSTG &&
              !wait_bounded(bar_empty + 8 * s, (ph - 1) & 1, abort_flag, g.status, tlim)) {
            stop = true;
            break;
          }
          const int seg = kb < g.nkb0 ? 0 : 1;
          const int kk = (seg ? kb - g.nkb0 : kb) * TBK;
          const CUtensorMap* ma = seg ? &mA1 : &mA0;
          const CUtensorMap* mb = seg ? &mB1 : &mB0;
          const uint32_t sA = ring + s * C::STAGE, sB = sA + C::TILE_A, fb = bar_full + 8 * s;
          mbar_arrive_expect_tx(fb, C::STAGE);
          const int ka = (seg ? g.ka0[1] : g.ka0[0]) + kk;
          const int kq = (seg ? g.kb0[1] : g.kb0[0]) + kk;
          if (A_MN) {  // 64(M) x 64(K) boxes
            tma_load_2d(sA, ma, mA, ka, fb);
            tma_load_2d(sA + 8192, ma, mA + 64, ka, fb);
          } else {  // one 64(K) x 128(M) box
            tma_load_2d(sA, ma, ka, mA, fb);
          }
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) tma_load_2d(sB + j * 8192, mb, nB + 64 * j, kq, fb);
          } else {  // one 64(K) x BN box
            tma_load_2d(sB, mb, kq, nB, fb);
          }
        }
      }
      issued_s = it;
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(TBM, BN, A_MN, B_MN);
      int it = 0, i = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < nunits && !stop; u += gridDim.x, ++i) {
        const Unit w = unit_of(g, u);
        const int a = i & 1;
        // the epilogue has drained this accumulator buffer (unit i - 2)
        if (i >= 2 &&
            !wait_bounded(bar_tempty + 8 * a, ((i >> 1) - 1) & 1, abort_flag, g.status, tlim))
          break;
        tc_fence_after();
        const uint32_t dacc = tmem + (uint32_t)(a * BN);
        for (int kb = w.kb_lo; kb < w.kb_hi; ++kb, ++it) {
          const int s = it % NSTG, ph = it / NSTG;
          if (!wait_bounded(bar_full + 8 * s, ph & 1, abort_flag, g.status, tlim)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t sA = ring + s * C::STAGE, sB = sA + C::TILE_A;
#pragma unroll
          for (int k4 = 0; k4 < TBK / 16; ++k4) {
            // K step of 16: 32 bytes along a K-major row, 16 rows (2048 B) of an MN-major tile
            const uint64_t ad = A_MN ? sdesc_sw128(sA + k4 * 2048, 8192, 1024)
                                     : sdesc_sw128(sA + k4 * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(sB + k4 * 2048, 8192, 1024)
                                     : sdesc_sw128(sB + k4 * 32, 16, 1024);
            umma_bf16(dacc, ad, bd, idesc, (kb != w.kb_lo || k4 != 0) ? 1u : 0u);
          }
          umma_commit(bar_empty + 8 * s);  // stage reusable once these MMAs are done
        }
        umma_commit(bar_tfull + 8 * a);  // this unit's MMAs complete -> epilogue
      }
      consumed_s = it;
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int i = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++i) {
      const Unit w = unit_of(g, u);
      const int a = i & 1;
      if (!wait_bounded(bar_tfull + 8 * a, (i >> 1) & 1, abort_flag, g.status, tlim)) break;
      tc_fence_after();
      const int row = w.m_base + q * 32 + lane;
      const bool row_ok = row < g.M;
      const bool empty_k = w.kb_hi == w.kb_lo;
      const int n_base = w.n_base * BN;
      if constexpr (OUT == kOutBf16Bias) {
        epilogue_bf16_bias<BN>(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * BN), g.bias,
                               n_base, g.N, w.m_base + q * 32, g.M, empty_k,
                               out_stage + (uint32_t)q * 8192, bias_s + (uint32_t)q * 128, &mC);
      } else {
      float* cf = static_cast<float*>(g.C) + w.z * g.c_stride_z + (size_t)row * g.ldc;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];  // columns n_base + 32c .. + 31 of this thread's row
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * BN + c * 32), r);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n0 = n_base + c * 32 + h * 16;
          if (!row_ok || n0 >= g.N) continue;
          uint32_t* v = r + 16 * h;
          if (empty_k) {  // no k blocks: the sum is zero
            if constexpr (OUT == kOutF32Add) {
              continue;
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = 0u;
            }
          }
          if (OUT == kOutF32) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(cf + n0 + j), "r"(v[j]),
                           "r"(v[j + 1]), "r"(v[j + 2]), "r"(v[j + 3])
                           : "memory");
          } else {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              asm volatile("red.global.add.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(cf + n0 + j),
                           "f"(__uint_as_float(v[j])), "f"(__uint_as_float(v[j + 1])),
                           "f"(__uint_as_float(v[j + 2])), "f"(__uint_as_float(v[j + 3]))
                           : "memory");
          }
        }
      }
      }
      // accumulator buffer a may be overwritten by unit i + 2
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * a);
    }
  }

  if (OUT == kOutBf16Bias && warp >= 2 && lane == 0) bulk_wait_all();  // output stores done
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    if (lane == 0 && *abort_flag) {
      // let TMA copies that were issued but never consumed land before exit
      for (int k = consumed_s; k < issued_s; ++k) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar_full + 8 * (k % NSTG), (k / NSTG) & 1))
          if (globaltimer_ns() - t0 > 10000000ull) break;
      }
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

// ------------------------------------------------------------ host side --
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 row-major [rows, cols] with a row pitch in elements; box {bx cols, by rows}
int make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t pitch,
             uint32_t bx, uint32_t by) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return (int)cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch * 2};
  const cuuint32_t box[2] = {bx, by};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

namespace {

// grid: one CTA per SM (at most one per unit, at most max_ctas if > 0)
template <bool A_MN, bool B_MN, int OUT, int BN>
int launch_tc(const CUtensorMap& a0, const CUtensorMap& b0, const CUtensorMap& a1,
              const CUtensorMap& b1, const CUtensorMap& c, GemmArgs g, cudaStream_t s,
              int max_ctas = 0) {
  using C = TcCfg<BN, OUT>;
  auto kern = tc_gemm_kernel<A_MN, B_MN, OUT, BN>;
  static int prepared[64][5];
  const int e = prepare_launch(prepared, kern, C::SMEM, 192, 1);
  if (e != 0) return e;
  g.tiles_m = (g.M + TBM - 1) / TBM;
  g.tiles_n = (g.N + BN - 1) / BN;
  const long long units = (long long)g.Z * g.tiles_m * g.tiles_n * g.ksplit;
  if (units > 0x7fffffffLL) return (int)cudaErrorInvalidValue;
  int cap = num_sms();
  if (max_ctas > 0 && max_ctas < cap) cap = max_ctas;
  const int grid = (int)(units < cap ? units : cap);
  if (grid == 0) return 0;
  kern<<<grid, 192, C::SMEM, s>>>(a0, b0, a1, b1, c, g);
  return (int)cudaGetLastError();
}

}  // namespace

int sm_count() { return num_sms(); }

int launch_dR_tc(const void* h_seq, const void* h0b, const void* dG, float* dR, int T, int B,
                 int NH, int Dh, int G, int* status, unsigned long long timeout_ns,
                 cudaStream_t s) {
  const int GD = G * Dh;
  CUtensorMap a0, a1, b0;
  int e = make_map(&a0, h0b, (uint64_t)B, (uint64_t)NH * Dh, (uint64_t)NH * Dh, 64, 64);
  if (e) return e;
  e = make_map(&b0, dG, (uint64_t)T * B, (uint64_t)NH * GD, (uint64_t)NH * GD, 64, 64);
  if (e) return e;
  a1 = a0;
  if (T > 1) {
    e = make_map(&a1, h_seq, (uint64_t)(T - 1) * B, (uint64_t)NH * Dh, (uint64_t)NH * Dh, 64, 64);
    if (e) return e;
  }
  GemmArgs g{};
  g.M = Dh;
  g.N = GD;
  g.Z = NH;
  g.m_off_z = Dh;
  g.n_off_z = GD;
  g.nkb0 = (B + TBK - 1) / TBK;
  g.nkb1 = T > 1 ? ((T - 1) * B + TBK - 1) / TBK : 0;
  g.ka0[0] = 0;
  g.ka0[1] = 0;
  g.kb0[0] = 0;
  g.kb0[1] = B;  // dG row of (t = 1, b = 0): pairs with h_0 = h_seq row 0
  g.C = dR;
  g.c_stride_z = (long long)Dh * GD;
  g.ldc = GD;
  g.bias = nullptr;
  g.status = status;
  g.timeout_ns = timeout_ns;
  // split K (= T*B rows) until the tiles cover the SMs, keeping >= 16 k blocks per split
  const int tiles = NH * ((Dh + TBM - 1) / TBM) * ((GD + 255) / 256);
  const int nkb = g.nkb0 + g.nkb1;
  int ks = num_sms() / (tiles > 0 ? tiles : 1);
  if (ks > nkb / 16) ks = nkb / 16;
  g.ksplit = ks > 1 ? ks : 1;
  if (g.ksplit == 1) return launch_tc<true, true, kOutF32, 256>(a0, b0, a1, b0, a0, g, s);
  if (cudaMemsetAsync(dR, 0, (size_t)NH * Dh * GD * sizeof(float), s) != cudaSuccess)
    return (int)cudaErrorInvalidValue;
  return launch_tc<true, true, kOutF32Add, 256>(a0, b0, a1, b0, a0, g, s);
}

int launch_input_proj_tc(const void* x, const void* W, const float* bias, void* Wx, int M, int N,
                         int K, int* status, unsigned long long timeout_ns, cudaStream_t s,
                         int max_ctas) {
  const bool wide = N >= 256;
  if (wide) {  // 256 x 256 tiles on CTA pairs, unless no pair can be launched here
    const int e = launch_input_proj_pair(x, W, bias, Wx, M, N, K, status, timeout_ns, s, max_ctas);
    if (e != -1) return e;
  }
  CUtensorMap a0, b0, c0;
  int e = make_map(&a0, x, (uint64_t)M, (uint64_t)K, (uint64_t)K, 64, 128);
  if (e) return e;
  e = make_map(&b0, W, (uint64_t)N, (uint64_t)K, (uint64_t)K, 64, wide ? 256 : 128);
  if (e) return e;
  e = make_map(&c0, Wx, (uint64_t)M, (uint64_t)N, (uint64_t)N, 64, 32);  // output boxes
  if (e) return e;
  GemmArgs g{};
  g.M = M;
  g.N = N;
  g.Z = 1;
  g.ksplit = 1;
  g.nkb0 = (K + TBK - 1) / TBK;
  g.nkb1 = 0;
  g.C = Wx;
  g.c_stride_z = 0;
  g.ldc = N;
  g.bias = bias;
  g.status = status;
  g.timeout_ns = timeout_ns;
  if (wide) return launch_tc<false, false, kOutBf16Bias, 256>(a0, b0, a0, b0, c0, g, s, max_ctas);
  return launch_tc<false, false, kOutBf16Bias, 128>(a0, b0, a0, b0, c0, g, s, max_ctas);
}

}  // namespace srnn
