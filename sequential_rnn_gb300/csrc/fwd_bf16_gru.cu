// bf16 forward instantiations for the GRU cell (see fwd_bf16.cuh).
#include "fwd_bf16.cuh"

namespace srnn {

int launch_fwd_bf16_gru(const FwdParams& p, int Dh, int NT, cudaStream_t s, bool query_only,
                        LaunchInfo* info) {
  // <cell, Dh, units per warp, n-tiles, KREG = k16 steps of R^T held in registers>
  if (NT != 1) return (int)cudaErrorInvalidValue;
  switch (Dh) {
    // slices of up to 64 units: 8 units per warp (24 gate rows padded to 2 m16
    // tiles), spreading a slice over more warps; larger slices keep 16 (the
    // register budget and R on chip)
    case 32: return launch_fwd_bf16_t<kGRU, 32, 8, 1, 2>(p, s, query_only, info);
    case 64: return launch_fwd_bf16_t<kGRU, 64, 8, 1, 4>(p, s, query_only, info);
    case 128:
      if (p.U <= 64) return launch_fwd_bf16_t<kGRU, 128, 8, 1, 8>(p, s, query_only, info);
      return launch_fwd_bf16_t<kGRU, 128, 16, 1, 6>(p, s, query_only, info);
    case 256: return launch_fwd_bf16_t<kGRU, 256, 16, 1, 10>(p, s, query_only, info);
    case 768: return launch_fwd_bf16_t<kGRU, 768, 16, 1, 10>(p, s, query_only, info);
    default: return (int)cudaErrorInvalidValue;
  }
}


// the same variants' launch limits, for the plan search
int fwd_bf16_gru_limits(int Dh, int U, FwdLimits* o) {
  switch (Dh) {
    case 32: fwd_bf16_limits_t<kGRU, 32, 8, 1, 2>(U, o); return 0;
    case 64: fwd_bf16_limits_t<kGRU, 64, 8, 1, 4>(U, o); return 0;
    case 128:
      if (U <= 64) fwd_bf16_limits_t<kGRU, 128, 8, 1, 8>(U, o);
      else fwd_bf16_limits_t<kGRU, 128, 16, 1, 6>(U, o);
      return 0;
    case 256: fwd_bf16_limits_t<kGRU, 256, 16, 1, 10>(U, o); return 0;
    case 768: fwd_bf16_limits_t<kGRU, 768, 16, 1, 10>(U, o); return 0;
    default: return 1;
  }
}

}  // namespace srnn
