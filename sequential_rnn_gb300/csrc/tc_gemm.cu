// Dense bf16 GEMMs of the path on the 5th-generation tensor cores:
//
//   dR[h] = sum_{t,b} h_{t-1}[b,h,:]^T dG_t[b,h,:]          (weight gradient)
//   Wx    = x W^T + b                                       (input projection)
//
// One 128 x 128 fp32 output tile per CTA, accumulated in tensor memory by
// tcgen05.mma (M=128, N=128, K=16 per instruction) from 128-byte-swizzled
// shared-memory tiles that TMA loads through a 6-stage ring:
//   warp 0   TMA producer (one lane) and TMEM owner (alloc / dealloc),
//   warp 1   MMA issuer (one lane): 4 MMAs per 64-deep k block, then a
//            tcgen05.commit that frees the ring stage once they completed,
//   warps 2-5 epilogue: tcgen05.ld of their 32-lane TMEM quarter (one output
//            row per thread), then fp32 or bf16(+bias) stores.
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

namespace srnn {
namespace {

constexpr int TBM = 128, TBN = 128, TBK = 64, TSTG = 6;
constexpr uint32_t TILE_A = TBM * TBK * 2;  // 16 KB
constexpr uint32_t TILE_B = TBN * TBK * 2;  // 16 KB
constexpr uint32_t STAGE_BYTES = TILE_A + TILE_B;
constexpr uint32_t TMEM_COLS = 128;
// ring + 1024 for aligning it + barriers (full, empty, accumulator) and the TMEM slot
constexpr uint32_t SMEM_BYTES = TSTG * STAGE_BYTES + 1024 + (2 * TSTG + 2) * 8 + 16;

enum : int { kOutF32 = 0, kOutBf16Bias = 1 };

struct GemmArgs {
  int M, N;                // valid output rows / columns per batch item z
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

template <bool A_MN, bool B_MN, int OUT>
__global__ void __launch_bounds__(192, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mB0,
                   const __grid_constant__ CUtensorMap mA1, const __grid_constant__ CUtensorMap mB1,
                   const GemmArgs g) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ int abort_flag_s;
  __shared__ int consumed_s, issued_s;
  volatile int* abort_flag = &abort_flag_s;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;  // 128-byte swizzle: 1024-byte aligned tiles
  const uint32_t bar_full = ring + TSTG * STAGE_BYTES, bar_empty = bar_full + 8 * TSTG;
  const uint32_t bar_acc = bar_empty + 8 * TSTG, tslot = bar_acc + 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int z = blockIdx.z, m_base = blockIdx.y * TBM, n_base = blockIdx.x * TBN;
  const int nkb = g.nkb0 + g.nkb1;

  if (threadIdx.x == 32) {
    for (int s = 0; s < TSTG; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc, 1);
    abort_flag_s = 0;
    consumed_s = 0;
    issued_s = 0;
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(tslot, TMEM_COLS);
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
      const int mA = m_base + z * g.m_off_z, nB = n_base + z * g.n_off_z;
      int kb = 0;
      for (; kb < nkb; ++kb) {
        const int s = kb % TSTG, u = kb / TSTG;
        if (kb >= TSTG && !wait_bounded(bar_empty + 8 * s, (u - 1) & 1, abort_flag, g.status, tlim))
          break;
        const int seg = kb < g.nkb0 ? 0 : 1;
        const int kk = (seg ? kb - g.nkb0 : kb) * TBK;
        const CUtensorMap* ma = seg ? &mA1 : &mA0;
        const CUtensorMap* mb = seg ? &mB1 : &mB0;
        const uint32_t sA = ring + s * STAGE_BYTES, sB = sA + TILE_A, fb = bar_full + 8 * s;
        mbar_arrive_expect_tx(fb, STAGE_BYTES);
        const int ka = (seg ? g.ka0[1] : g.ka0[0]) + kk, kbq = (seg ? g.kb0[1] : g.kb0[0]) + kk;
        if (A_MN) {  // two 64(M) x 64(K) boxes
          tma_load_2d(sA, ma, mA, ka, fb);
          tma_load_2d(sA + TILE_A / 2, ma, mA + 64, ka, fb);
        } else {  // one 64(K) x 128(M) box
          tma_load_2d(sA, ma, ka, mA, fb);
        }
        if (B_MN) {
          tma_load_2d(sB, mb, nB, kbq, fb);
          tma_load_2d(sB + TILE_B / 2, mb, nB + 64, kbq, fb);
        } else {
          tma_load_2d(sB, mb, kbq, nB, fb);
        }
      }
      issued_s = kb;
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(TBM, TBN, A_MN, B_MN);
      int kb = 0;
      for (; kb < nkb; ++kb) {
        const int s = kb % TSTG, u = kb / TSTG;
        if (!wait_bounded(bar_full + 8 * s, u & 1, abort_flag, g.status, tlim)) break;
        tc_fence_after();
        const uint32_t sA = ring + s * STAGE_BYTES, sB = sA + TILE_A;
#pragma unroll
        for (int k4 = 0; k4 < TBK / 16; ++k4) {
          // K step of 16: 32 bytes along a K-major row, 16 rows (2048 B) of an MN-major tile
          const uint64_t ad = A_MN ? sdesc_sw128(sA + k4 * 2048, TILE_A / 2, 1024)
                                   : sdesc_sw128(sA + k4 * 32, 16, 1024);
          const uint64_t bd = B_MN ? sdesc_sw128(sB + k4 * 2048, TILE_B / 2, 1024)
                                   : sdesc_sw128(sB + k4 * 32, 16, 1024);
          umma_bf16(tmem, ad, bd, idesc, (kb | k4) != 0);
        }
        umma_commit(bar_empty + 8 * s);  // stage reusable once these MMAs are done
      }
      consumed_s = kb;
      umma_commit(bar_acc);  // every issued MMA complete -> accumulator ready
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const bool ok = wait_bounded(bar_acc, 0, abort_flag, g.status, tlim);
    tc_fence_after();
    const int row = m_base + q * 32 + lane;
    const bool row_ok = ok && !*abort_flag && row < g.M;
#pragma unroll 1
    for (int c = 0; c < TBN / 16; ++c) {
      uint32_t r[16];
      tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 16), r);
      tmem_wait_ld();
      const int n0 = n_base + c * 16;
      if (!row_ok || n0 >= g.N) continue;
      if (nkb == 0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = 0u;
      }
      if (OUT == kOutF32) {
        float* dst = static_cast<float*>(g.C) + z * g.c_stride_z + (size_t)row * g.ldc + n0;
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(dst + j), "r"(r[j]),
                       "r"(r[j + 1]), "r"(r[j + 2]), "r"(r[j + 3])
                       : "memory");
      } else {
        __nv_bfloat16* dst =
            static_cast<__nv_bfloat16*>(g.C) + z * g.c_stride_z + (size_t)row * g.ldc + n0;
        uint32_t pk[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float a = __uint_as_float(r[2 * j]), b = __uint_as_float(r[2 * j + 1]);
          if (g.bias) {
            a += g.bias[n0 + 2 * j];
            b += g.bias[n0 + 2 * j + 1];
          }
          pk[j] = pack_bf16x2(a, b);
        }
#pragma unroll
        for (int j = 0; j < 8; j += 4)
          asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(dst + 2 * j), "r"(pk[j]),
                       "r"(pk[j + 1]), "r"(pk[j + 2]), "r"(pk[j + 3])
                       : "memory");
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    if (lane == 0 && *abort_flag) {
      // let TMA copies that were issued but never consumed land before exit
      for (int kb = consumed_s; kb < issued_s; ++kb) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar_full + 8 * (kb % TSTG), (kb / TSTG) & 1))
          if (globaltimer_ns() - t0 > 10000000ull) break;
      }
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

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

template <bool A_MN, bool B_MN, int OUT>
int launch_tc(const CUtensorMap& a0, const CUtensorMap& b0, const CUtensorMap& a1,
              const CUtensorMap& b1, const GemmArgs& g, int Z, cudaStream_t s) {
  auto kern = tc_gemm_kernel<A_MN, B_MN, OUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return (int)e;
  const dim3 grid((g.N + TBN - 1) / TBN, (g.M + TBM - 1) / TBM, Z);
  kern<<<grid, 192, SMEM_BYTES, s>>>(a0, b0, a1, b1, g);
  return (int)cudaGetLastError();
}

}  // namespace

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
  return launch_tc<true, true, kOutF32>(a0, b0, a1, b0, g, NH, s);
}

int launch_input_proj_tc(const void* x, const void* W, const float* bias, void* Wx, int M, int N,
                         int K, int* status, unsigned long long timeout_ns, cudaStream_t s) {
  CUtensorMap a0, b0;
  int e = make_map(&a0, x, (uint64_t)M, (uint64_t)K, (uint64_t)K, 64, 128);
  if (e) return e;
  e = make_map(&b0, W, (uint64_t)N, (uint64_t)K, (uint64_t)K, 64, 128);
  if (e) return e;
  GemmArgs g{};
  g.M = M;
  g.N = N;
  g.nkb0 = (K + TBK - 1) / TBK;
  g.nkb1 = 0;
  g.C = Wx;
  g.c_stride_z = 0;
  g.ldc = N;
  g.bias = bias;
  g.status = status;
  g.timeout_ns = timeout_ns;
  return launch_tc<false, false, kOutBf16Bias>(a0, b0, a0, b0, g, 1, s);
}

}  // namespace srnn
