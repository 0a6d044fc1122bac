// bf16 forward instantiations for the sLSTM cell (see fwd_bf16.cuh).
#include "fwd_bf16.cuh"

namespace srnn {

int launch_fwd_bf16_slstm(const FwdParams& p, int Dh, int NT, int hsplit, cudaStream_t s,
                          bool query_only, LaunchInfo* info) {
  // <cell, Dh, units per warp, n-tiles, KREG = k16 steps of R^T held in registers, HS>
  if (NT != 1) return (int)cudaErrorInvalidValue;
  if (hsplit == 2) {
    // the hi + lo pair in one n8 tile (batch slices of 4 rows): half the MMAs
    switch (Dh) {
      case 32: return launch_fwd_bf16_t<kSLSTM, 32, 8, 1, 2, 2>(p, s, query_only, info);
      case 64: return launch_fwd_bf16_t<kSLSTM, 64, 8, 1, 4, 2>(p, s, query_only, info);
      case 128: return launch_fwd_bf16_t<kSLSTM, 128, 8, 1, 8, 2>(p, s, query_only, info);
      case 256: return launch_fwd_bf16_t<kSLSTM, 256, 8, 1, 14, 2>(p, s, query_only, info);
      default: return (int)cudaErrorInvalidValue;
    }
  }
  if (hsplit) {
    // h_{t-1} as a bf16 hi + lo pair: the exponentially gated recurrence amplifies
    // per-step rounding of h by orders of magnitude over thousands of steps.
    switch (Dh) {
      case 32: return launch_fwd_bf16_t<kSLSTM, 32, 8, 1, 2, 1>(p, s, query_only, info);
      case 64: return launch_fwd_bf16_t<kSLSTM, 64, 8, 1, 4, 1>(p, s, query_only, info);
      case 128: return launch_fwd_bf16_t<kSLSTM, 128, 8, 1, 8, 1>(p, s, query_only, info);
      case 256: return launch_fwd_bf16_t<kSLSTM, 256, 8, 1, 12, 1>(p, s, query_only, info);
      default: return (int)cudaErrorInvalidValue;
    }
  }
  switch (Dh) {
    case 32: return launch_fwd_bf16_t<kSLSTM, 32, 8, 1, 2>(p, s, query_only, info);
    case 64: return launch_fwd_bf16_t<kSLSTM, 64, 8, 1, 4>(p, s, query_only, info);
    case 128: return launch_fwd_bf16_t<kSLSTM, 128, 8, 1, 8>(p, s, query_only, info);
    case 256: return launch_fwd_bf16_t<kSLSTM, 256, 8, 1, 16>(p, s, query_only, info);
    case 768: return launch_fwd_bf16_t<kSLSTM, 768, 8, 1, 18>(p, s, query_only, info);
    default: return (int)cudaErrorInvalidValue;
  }
}


// the same variants' launch limits, for the plan search
int fwd_bf16_slstm_limits(int Dh, int hsplit, int U, FwdLimits* o) {
  if (hsplit == 2) {
    switch (Dh) {
      case 32: fwd_bf16_limits_t<kSLSTM, 32, 8, 1, 2, 2>(U, o); return 0;
      case 64: fwd_bf16_limits_t<kSLSTM, 64, 8, 1, 4, 2>(U, o); return 0;
      case 128: fwd_bf16_limits_t<kSLSTM, 128, 8, 1, 8, 2>(U, o); return 0;
      case 256: fwd_bf16_limits_t<kSLSTM, 256, 8, 1, 14, 2>(U, o); return 0;
      default: return 1;
    }
  }
  if (hsplit) {
    switch (Dh) {
      case 32: fwd_bf16_limits_t<kSLSTM, 32, 8, 1, 2, 1>(U, o); return 0;
      case 64: fwd_bf16_limits_t<kSLSTM, 64, 8, 1, 4, 1>(U, o); return 0;
      case 128: fwd_bf16_limits_t<kSLSTM, 128, 8, 1, 8, 1>(U, o); return 0;
      case 256: fwd_bf16_limits_t<kSLSTM, 256, 8, 1, 12, 1>(U, o); return 0;
      default: return 1;
    }
  }
  switch (Dh) {
    case 32: fwd_bf16_limits_t<kSLSTM, 32, 8, 1, 2>(U, o); return 0;
    case 64: fwd_bf16_limits_t<kSLSTM, 64, 8, 1, 4>(U, o); return 0;
    case 128: fwd_bf16_limits_t<kSLSTM, 128, 8, 1, 8>(U, o); return 0;
    case 256: fwd_bf16_limits_t<kSLSTM, 256, 8, 1, 16>(U, o); return 0;
    case 768: fwd_bf16_limits_t<kSLSTM, 768, 8, 1, 18>(U, o); return 0;
    default: return 1;
  }
}

}  // namespace srnn
