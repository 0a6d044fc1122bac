// Internal interface of the C-ABI library (not installed): the helpers the
// single-call entry points (capi.cu), the launch-plan search (plan.cu) and the
// multi-launch runtimes (runtime.cu) share.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/rnn.h"
#include "kernels.h"

namespace srnn {
namespace api {

constexpr size_t kStatusBytes = 256;                          // status word + padding
constexpr unsigned long long kTimeoutNs = 2000000000ull;      // 2 s per device wait
constexpr unsigned long long kTestTimeoutNs = 50000000ull;    // 50 ms under the test flag
constexpr int kMaxLayers = 8;                                 // stacked layers per call
constexpr int kSlstmPlainMaxT = 768;  // longest sLSTM (Dh > 256) sequence without RNN_FLAG_H_BF16

inline int gates_of(int cell) { return cell == RNN_GRU ? 3 : 4; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
// fp32 state arrays a cell carries: LSTM h, c; GRU h; sLSTM h, c, n, m
inline int state_arrays(int cell) { return cell == RNN_LSTM ? 2 : (cell == RNN_GRU ? 1 : 4); }

int check_desc(const rnn_desc_t* d);
// sLSTM h operand of the bf16 forward: 0 bf16, 1 hi + lo operands, 2 hi + lo in one n8 tile
int hsplit_mode(const rnn_desc_t* d);
bool bf16_dh_supported(int Dh);

// Launch plan of one forward: fp32 or bf16 path, CTAs per head (CS), units per
// CTA (U), n-tiles and batch rows per CTA, batch slices.
struct Plan {
  bool f32;
  int CS, U, NT, NB, nbslices;
};
// Result of the plan search: CTAs per head, time chunk, CTAs per layer, waves
// over the SMs, predicted time (microseconds).
struct PlanChoice {
  int cs, chunk, ctas, waves;
  double us;
};

int device_sms();
// Planned time of one recurrence step (ns) of the bf16 forward with CS CTAs per
// head (measured table, else the latency model); 0 when no variant fits.
double plan_step_ns(const rnn_desc_t* d, int cs);
// L = 1: one forward over T steps; L > 1: the stacked wavefront (chunk_req 0 =
// choose the chunk).  d->cluster != 0 restricts the search to that size.
int plan_search(const rnn_desc_t* d, int L, int sms, int chunk_req, PlanChoice* out);
int make_plan(const rnn_desc_t* d, Plan* pl);
int map_launch_error(int e);
int launch_forward(const rnn_desc_t* d, const Plan& pl, const FwdParams& p, cudaStream_t s,
                   bool query_only, LaunchInfo* info);
FwdParams base_params(const rnn_desc_t* d, const Plan& pl);
// Final state <- initial state (or zero) for a zero-length sequence.
int copy_state(float* dst, const float* src, size_t n, cudaStream_t s);
int clear_status(void* workspace, size_t workspace_bytes, cudaStream_t s);

}  // namespace api
}  // namespace srnn
