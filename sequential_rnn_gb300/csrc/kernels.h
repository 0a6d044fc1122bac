// Internal interface between the C ABI (capi.cu) and the kernel translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace srnn {

// Once-per-device preparation of a kernel's launches: dynamic shared memory and
// non-portable cluster-size attributes, and for clusters the co-scheduling
// check.  Cached per (device, cluster size) in `state` (0 = not prepared,
// 1 = ready, -1 = the cluster cannot be co-scheduled, else 1000 + CUDA error),
// so launches after the first make no driver queries.  Preparing twice is
// harmless, so concurrent first calls need no lock.
template <class Kern>
inline int prepare_launch(int (&state)[64][5], Kern kern, uint32_t smem, int threads, int cs) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return (int)cudaErrorInvalidDevice;
  const int ci = cs <= 1 ? 0 : cs == 2 ? 1 : cs == 4 ? 2 : cs == 8 ? 3 : 4;
  const bool cache = dev >= 0 && dev < 64;
  if (cache && state[dev][ci] != 0)
    return state[dev][ci] == 1 ? 0 : (state[dev][ci] == -1 ? -1 : state[dev][ci] - 1000);
  int r = 0, max_smem = 0;
  cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (smem > (uint32_t)max_smem) r = (int)cudaErrorInvalidConfiguration;
  // the attribute is per kernel, shared by every cluster size (each with its own
  // shared-memory need): allow all the device's opt-in amount the kernel's
  // static shared memory leaves
  if (r == 0) {
    cudaFuncAttributes fa;
    r = (int)cudaFuncGetAttributes(&fa, kern);
    if (r == 0 && smem + fa.sharedSizeBytes > (size_t)max_smem) r = (int)cudaErrorInvalidConfiguration;
    if (r == 0)
      r = (int)cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    max_smem - (int)fa.sharedSizeBytes);
  }
  if (r == 0 && cs > 8)
    r = (int)cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (r == 0 && cs > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int ncl = 0;
    r = (int)cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg);
    if (r == 0 && ncl < 1) r = -1;  // the cluster cannot be co-scheduled
  }
  if (cache) state[dev][ci] = r == 0 ? 1 : (r == -1 ? -1 : r + 1000);
  return r;
}

enum : int { kLSTM = 0, kGRU = 1, kSLSTM = 2 };
// bits of the device status word: a bounded wait ran out; (bounds-check builds)
// an index fell outside its buffer
enum : int { kStatusTimeout = 1, kStatusBounds = 2 };

// Arguments of one forward launch.  Grid: one CTA per (head, batch slice,
// cluster rank); blockIdx.x = ((head * nbslices) + bslice) * CS + rank.
struct FwdParams {
  const void* Wx;
  const void* R;
  const float* bias;
  const float* h0;
  const float* c0;
  const float* n0;
  const float* m0;
  void* h_seq;
  float* hT;
  float* cT;
  float* nT;
  float* mT;
  float* stash_gates;  // training stash: four gate values per cell   [T,B,NH,4Dh]
  float* stash_c;      // LSTM / sLSTM c_t, GRU h_t                     [T,B,NH,Dh]
  float* stash_n;      // sLSTM n_t                                     [T,B,NH,Dh]
  int* status;
  int T, B, NH;
  int CS;        // CTAs per (head, batch slice): thread-block cluster size
  int U;         // hidden units owned by one CTA (Dh / CS)
  int nbslices;  // batch slices per head
  int flags;
  unsigned long long timeout_ns;
};

struct LaunchInfo {
  int grid, threads, cluster, nb, smem, kernel_id;
};

// Each returns a cudaError_t value (cast to int); `info` is filled when non-null.
// With `query_only` nothing is launched.
int launch_fwd_f32(const FwdParams& p, int cell, int Dh, cudaStream_t s, bool query_only,
                   LaunchInfo* info);
// Launch limits of the compiled bf16 forward variant for (cell, Dh) (host only).
struct FwdLimits {
  int max_threads;     // CTA size the register budget allows
  int unit_group;      // hidden units per warp
  uint32_t smem;       // dynamic shared memory of a CTA owning U units
};
// each returns 0, or nonzero when no variant exists for Dh
int fwd_bf16_lstm_limits(int Dh, int U, FwdLimits* o);
int fwd_bf16_gru_limits(int Dh, int U, FwdLimits* o);
int fwd_bf16_slstm_limits(int Dh, int hsplit, int U, FwdLimits* o);

int launch_fwd_bf16_lstm(const FwdParams& p, int Dh, int NT, cudaStream_t s, bool query_only,
                         LaunchInfo* info);
int launch_fwd_bf16_gru(const FwdParams& p, int Dh, int NT, cudaStream_t s, bool query_only,
                        LaunchInfo* info);
// hsplit: h_{t-1} as a bf16 hi + lo pair and accurate gate math (sLSTM only):
// 1 = two B operands, 2 = both halves of one n8 tile (4 batch rows per CTA)
int launch_fwd_bf16_slstm(const FwdParams& p, int Dh, int NT, int hsplit, cudaStream_t s,
                          bool query_only, LaunchInfo* info);
// Units handled by one warp in the bf16 kernels (gate rows of one warp = UG * G).
// hidden units per warp of the bf16 forward variant for (cell, Dh, units per CTA)
inline int bf16_unit_group(int cell, int Dh, int U) {
  return cell == kGRU && (Dh > 128 || U > 64) ? 16 : 8;
}

// Empty-step kernel with the launch shape of a bf16/fp32 forward.
int launch_sync_floor(const LaunchInfo& li, int T, int* status, cudaStream_t s);

// Backward through time (bf16; LSTM, GRU, sLSTM).
struct BwdParams {
  const void* R;
  const void* dh_seq;
  const float* dhT;
  const float* dcT;    // LSTM / sLSTM
  const float* dnT;    // sLSTM
  const float* stash_gates;
  const float* stash_c;
  const float* stash_n;
  const float* h_init;  // h0 fp32 [B,NH,Dh] (GRU: h_{-1}); NULL = zeros
  const float* c_init;  // c0 fp32 (NULL = zeros), c_{-1} for the first step
  const float* n_init;  // sLSTM n0 (NULL = zeros)
  void* dWx;
  void* drec;           // GRU: recurrent-preactivation gradient, bf16 [T,B,NH,3Dh] (workspace)
  float* dh0;
  float* dc0;
  float* dn0;
  float* db_part;  // [nbslices, NH, G*Dh] per-slice bias-gradient partials (workspace)
  int* status;
  int T, B, NH;
  int CS, U, nbslices, flags;
  unsigned long long timeout_ns;
};
int launch_bwd_bf16(const BwdParams& p, int cell, int Dh, cudaStream_t s, bool query_only,
                    LaunchInfo* info);

// Weight-gradient helpers (grad_weights.cu): h0 -> bf16, db from per-slice partials.
int launch_h0_to_bf16(const float* h0, void* out, int n, cudaStream_t s);
// tcgen05 GEMMs (tc_gemm.cu).  dR[h] = sum_{t,b} h_{t-1}^T dG_t (fp32, overwritten),
// h_{-1} = h0b, dG [T,B,NH,G*Dh] bf16 (dWx for LSTM / sLSTM, the recurrent gradient
// for GRU); Wx = x W^T + bias (bf16).  status: device status word.
int launch_dR_tc(const void* h_seq, const void* h0b, const void* dG, float* dR, int T, int B,
                 int NH, int Dh, int G, int* status, unsigned long long timeout_ns,
                 cudaStream_t s);
// max_ctas > 0 caps the persistent grid (SMs left free for concurrent kernels)
int launch_input_proj_tc(const void* x, const void* W, const float* bias, void* Wx, int M, int N,
                         int K, int* status, unsigned long long timeout_ns, cudaStream_t s,
                         int max_ctas = 0);
int sm_count();
// CTA-pair input projection (tc_gemm_pair.cu), N >= 256: -1 when a pair cannot
// be launched (the caller takes the one-CTA kernel), else 0 or a CUDA error.
int launch_input_proj_pair(const void* x, const void* W, const float* bias, void* Wx, int M, int N,
                           int K, int* status, unsigned long long timeout_ns, cudaStream_t s,
                           int max_ctas);
int launch_db_reduce(const float* part, float* db, int nslices, int n, cudaStream_t s);

}  // namespace srnn
