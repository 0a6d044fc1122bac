// bf16 (+ bias) epilogue of the tcgen05 GEMMs, shared by the one-CTA and the
// CTA-pair kernels: one epilogue warp drains its 32 TMEM lanes (32 output rows)
// x BN accumulator columns.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"
#include "tc.cuh"

namespace srnn {

// Rows mr .. mr + 31, columns n_base .. n_base + BN - 1 of the output (M x N).
// tacc: TMEM address of this warp's lane quarter at the tile's first column.
// The values go through shared memory (`stg`, 8 KB: two 32-row x 64-column
// boxes in the 128-byte swizzled layout, 16-byte chunk j of row r at chunk
// j ^ (r % 8)) to TMA stores, 128 columns at a time; the TMA engine writes whole
// row segments and drops rows / columns past the output's extent.  The BN
// bias values are loaded once (lane i holds columns i, i + 32, ...; zeros past
// N or without a bias) and each 32-column slice passes through the warp's own
// 128-byte slot `bias_w` to be read as broadcasts (a global load per value and
// thread cost ~11 us of a 73 us projection, 16384 x 3072 x 768).
// empty_k: the sum had no k blocks (the accumulator was never written).
template <int BN>
__device__ __forceinline__ void epilogue_bf16_bias(uint32_t tacc, const float* bias, int n_base,
                                                   int N, int mr, int M, bool empty_k,
                                                   uint32_t stg, uint32_t bias_w,
                                                   const CUtensorMap* mC) {
  const int lane = threadIdx.x & 31;
  const bool has_bias = bias != nullptr;
  float breg[BN / 32];
#pragma unroll
  for (int k = 0; k < BN / 32; ++k) {
    const int n = n_base + 32 * k + lane;
    breg[k] = (has_bias && n < N) ? __ldg(bias + n) : 0.f;
  }
#pragma unroll 1
  for (int hh = 0; hh < BN / 128; ++hh) {
    if (lane == 0) bulk_wait_read_all();  // the previous boxes left this buffer
    __syncwarp();
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];  // columns n_base + 128 hh + 32 c .. + 31 of this thread's row
      tmem_ld32(tacc + (uint32_t)(hh * 128 + c * 32), r);
      tmem_wait_ld();
      tmem_reg_fence(r);
      uint32_t pk[16];
      float bv[32];
      if (has_bias) {
        float bk = 0.f;  // breg[hh * 4 + c] (indices fixed per unrolled copy)
#pragma unroll
        for (int k = 0; k < BN / 32; ++k)
          if (k == hh * 4 + c) bk = breg[k];
        __syncwarp();  // the slot's previous values were read
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(bias_w + 4u * lane), "f"(bk) : "memory");
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                       : "=f"(bv[j]), "=f"(bv[j + 1]), "=f"(bv[j + 2]), "=f"(bv[j + 3])
                       : "r"(bias_w + 4u * (uint32_t)j)
                       : "memory");
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) bv[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float x0 = (empty_k ? 0.f : __uint_as_float(r[2 * j])) + bv[2 * j];
        const float x1 = (empty_k ? 0.f : __uint_as_float(r[2 * j + 1])) + bv[2 * j + 1];
        pk[j] = pack_bf16x2(x0, x1);
      }
      const uint32_t rowb = stg + (uint32_t)(c >> 1) * 4096 + (uint32_t)lane * 128;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t chunk = (uint32_t)(((c & 1) * 4 + k) ^ (lane & 7));
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(rowb + chunk * 16),
                     "r"(pk[4 * k]), "r"(pk[4 * k + 1]), "r"(pk[4 * k + 2]), "r"(pk[4 * k + 3])
                     : "memory");
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the TMA engine
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int nc = n_base + hh * 128 + b * 64;
        if (nc < N && mr < M) tma_store_2d(mC, nc, mr, stg + (uint32_t)b * 4096);
      }
      bulk_commit();
    }
  }
}

}  // namespace srnn

namespace srnn {

// One epilogue warp's 32 rows (mr .. mr + 31) x 128 columns (n0 .. n0 + 127) of
// the output, bf16 (+ bias): two 64-column boxes staged one after the other in
// the warp's 4 KB buffer `stg` (32 rows x 128 B, 16-byte chunk j of row r at
// chunk j ^ (r % 8)) and written by TMA stores.  The second box's accumulator
// columns are loaded from TMEM while the first is converted and stored.
// tacc: TMEM address of the warp's lane quarter at column n0's accumulator.
// The bias of each 32-column slice passes through the warp's 128-byte slot
// `bias_w` and is read back as broadcasts.
__device__ __forceinline__ void epilogue_bf16_bias_128(uint32_t tacc, const float* bias, int n0,
                                                       int N, int mr, int M, uint32_t stg,
                                                       uint32_t bias_w, const CUtensorMap* mC) {
  const int lane = threadIdx.x & 31;
  const bool has_bias = bias != nullptr;
  float breg[4];  // lane i: columns n0 + 32 k + i
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int n = n0 + 32 * k + lane;
    breg[k] = (has_bias && n < N) ? __ldg(bias + n) : 0.f;
  }
  // one 32-column slice: bias (through the warp's slot, read as broadcasts,
  // four values at a time) + accumulator -> 16 bf16 pairs at pk[off ..]
  auto slice = [&](const uint32_t (&v)[32], float bk, uint32_t (&pk)[32], int off) {
    if (has_bias) {
      __syncwarp();  // the slot's previous values were read
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(bias_w + 4u * lane), "f"(bk) : "memory");
      __syncwarp();
    }
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      float b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
      if (has_bias)
        asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(b0), "=f"(b1), "=f"(b2), "=f"(b3)
                     : "r"(bias_w + 4u * (uint32_t)j)
                     : "memory");
      pk[off + j / 2] = pack_bf16x2(__uint_as_float(v[j]) + b0, __uint_as_float(v[j + 1]) + b1);
      pk[off + j / 2 + 1] =
          pack_bf16x2(__uint_as_float(v[j + 2]) + b2, __uint_as_float(v[j + 3]) + b3);
    }
  };
  // box b (64 columns, packed in pk) -> staging buffer -> TMA store
  auto store_box = [&](const uint32_t (&pk)[32], int b) {
    if (lane == 0) bulk_wait_read_all();  // the previous box left the buffer
    __syncwarp();
    const uint32_t rowb = stg + (uint32_t)lane * 128;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t chunk = (uint32_t)(k ^ (lane & 7));
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(rowb + chunk * 16),
                   "r"(pk[4 * k]), "r"(pk[4 * k + 1]), "r"(pk[4 * k + 2]), "r"(pk[4 * k + 3])
                   : "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the TMA engine
    __syncwarp();
    if (lane == 0) {
      const int nc = n0 + 64 * b;
      if (nc < N && mr < M) tma_store_2d(mC, nc, mr, stg);
      bulk_commit();
    }
  };
  // TMEM loads run one 32-column slice ahead of the conversion
  uint32_t r0[32], r1[32], r2[32], r3[32], pk[32];
  tmem_ld32(tacc, r0);
  tmem_ld32(tacc + 32u, r1);
  tmem_wait_ld();
  tmem_reg_fence(r0);
  tmem_reg_fence(r1);
  tmem_ld32(tacc + 64u, r2);
  slice(r0, breg[0], pk, 0);
  slice(r1, breg[1], pk, 16);
  store_box(pk, 0);
  tmem_wait_ld();
  tmem_reg_fence(r2);
  tmem_ld32(tacc + 96u, r3);
  slice(r2, breg[2], pk, 0);
  tmem_wait_ld();
  tmem_reg_fence(r3);
  slice(r3, breg[3], pk, 16);
  store_box(pk, 1);
}

}  // namespace srnn
