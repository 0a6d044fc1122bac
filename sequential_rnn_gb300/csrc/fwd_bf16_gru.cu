// bf16 forward instantiations for the GRU cell (see fwd_bf16.cuh).
#include "fwd_bf16.cuh"

namespace srnn {

int launch_fwd_bf16_gru(const FwdParams& p, int Dh, int NT, cudaStream_t s, bool query_only,
                          LaunchInfo* info) {
  // KREG: k16 steps of R^T held in registers per warp; the rest sit in shared memory.
  constexpr int UG = 16;
  if (NT == 2) {
    switch (Dh) {
      case 32: return launch_fwd_bf16_t<kGRU, 32, UG, 2, 2>(p, s, query_only, info);
      case 64: return launch_fwd_bf16_t<kGRU, 64, UG, 2, 4>(p, s, query_only, info);
      case 128: return launch_fwd_bf16_t<kGRU, 128, UG, 2, 8>(p, s, query_only, info);
      default: return (int)cudaErrorInvalidValue;
    }
  }
  switch (Dh) {
    case 32: return launch_fwd_bf16_t<kGRU, 32, UG, 1, 2>(p, s, query_only, info);
    case 64: return launch_fwd_bf16_t<kGRU, 64, UG, 1, 4>(p, s, query_only, info);
    case 128: return launch_fwd_bf16_t<kGRU, 128, UG, 1, 6>(p, s, query_only, info);
    case 256: return launch_fwd_bf16_t<kGRU, 256, UG, 1, (UG == 16 ? 10 : 16)>(p, s, query_only, info);
    case 768: return launch_fwd_bf16_t<kGRU, 768, UG, 1, 10>(p, s, query_only, info);
    default: return (int)cudaErrorInvalidValue;
  }
}

}  // namespace srnn
