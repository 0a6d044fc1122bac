// C ABI of the head-wise RNN recurrence (declared in include/rnn.h):
// argument checks, kernel-variant selection, launch geometry and launches on
// the caller's stream.  The library allocates no device memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/rnn.h"
#include "kernels.h"

using namespace srnn;

namespace {

constexpr size_t kStatusBytes = 256;
constexpr unsigned long long kTimeoutNs = 2000000000ull;      // 2 s per wait
constexpr unsigned long long kTestTimeoutNs = 50000000ull;    // 50 ms under the test flag

int gates_of(int cell) { return cell == RNN_GRU ? 3 : 4; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int check_desc(const rnn_desc_t* d) {
  if (d == nullptr) return RNN_ERR_INVALID_ARG;
  if (d->cell < RNN_LSTM || d->cell > RNN_SLSTM) return RNN_ERR_INVALID_ARG;
  if (d->dtype != RNN_F32 && d->dtype != RNN_BF16) return RNN_ERR_INVALID_ARG;
  if (d->T < 0 || d->B < 0 || d->NH < 0 || d->Dh <= 0) return RNN_ERR_INVALID_ARG;
  if (d->cluster < 0) return RNN_ERR_INVALID_ARG;
  return RNN_OK;
}

// ------------------------------------------------------------ plan search --
// The launch plan (CTAs per head; for stacked layers also the time chunk) is an
// integer search in the spirit of the FlashRNN card's ConstrINT (hardware
// limits as integer constraints with divisibility): every candidate must
// divide the head into whole warps' unit groups, fit the compiled variant's
// register budget (threads per CTA) and shared memory; among the feasible ones
// the cost is the per-step time times the waves the CTAs need over the SMs
// (and, for a stack, how many layers' recurrences can be resident at once).
// Per-step times: measured on GB300 (bf16 forward, T = 512, inputs in L2), by
// CTAs per head 1, 2, 4, 8, 16; 0 = not measured -> model below.
struct StepRow {
  int cell, Dh;
  float ns[5];
};
const StepRow kStepTable[] = {
    {RNN_LSTM, 32, {332, 400, 388, 0, 0}},        {RNN_LSTM, 64, {438, 416, 405, 415, 0}},
    {RNN_LSTM, 128, {0, 533, 442, 455, 505}},     {RNN_LSTM, 256, {0, 0, 776, 617, 708}},
    {RNN_LSTM, 768, {0, 0, 0, 0, 1933}},          {RNN_GRU, 32, {334, 393, 0, 0, 0}},
    {RNN_GRU, 64, {377, 417, 428, 0, 0}},         {RNN_GRU, 128, {697, 506, 498, 509, 0}},
    {RNN_GRU, 256, {0, 970, 753, 715, 791}},      {RNN_GRU, 768, {0, 0, 0, 0, 1996}},
    {RNN_SLSTM, 32, {403, 452, 464, 0, 0}},       {RNN_SLSTM, 64, {571, 507, 510, 576, 0}},
    {RNN_SLSTM, 128, {0, 897, 679, 690, 727}},    {RNN_SLSTM, 256, {0, 0, 1425, 1128, 1172}},
    {RNN_SLSTM, 768, {0, 0, 0, 0, 2013}},
};
constexpr int kClusterSizes[5] = {1, 2, 4, 8, 16};
constexpr int kMaxSmemOptin = 232448;       // dynamic shared memory per CTA (sm_103)
constexpr double kChunkOverheadUs = 20.0;   // launch + prologue of one stacked chunk
constexpr double kProjTflops = 600.0;       // input-projection GEMM rate on all SMs (chunk sizes)

int log2_cs(int cs) { return cs == 1 ? 0 : cs == 2 ? 1 : cs == 4 ? 2 : cs == 8 ? 3 : 4; }

bool hsplit_of(const rnn_desc_t* d) {
  return d->cell == RNN_SLSTM && !(d->flags & RNN_FLAG_H_BF16) && d->Dh <= 256;
}

// Fallback model for unmeasured points: sync floor of the launch shape plus a
// fixed latency chain plus tensor-pipe issue (8-cycle mma.sync per sub-partition).
double model_step_ns(const rnn_desc_t* d, int cs, int unit_group) {
  const int G = gates_of(d->cell), U = d->Dh / cs, NW = U / unit_group;
  const int per_warp = unit_group * G / 16 * (d->Dh / 16) * (hsplit_of(d) ? 2 : 1);
  const double w = (double)per_warp * ((NW + 3) / 4);
  const double floor_ns = cs == 1 ? 160.0 : 205.0 + 4.0 * cs;
  return floor_ns + 150.0 + 7.0 * w;
}

bool cs_limits(const rnn_desc_t* d, int cs, FwdLimits* lim) {
  if (d->Dh % cs) return false;
  const int U = d->Dh / cs;
  int e = 1;
  if (d->cell == RNN_LSTM) e = fwd_bf16_lstm_limits(d->Dh, U, lim);
  else if (d->cell == RNN_GRU) e = fwd_bf16_gru_limits(d->Dh, U, lim);
  else e = fwd_bf16_slstm_limits(d->Dh, hsplit_of(d) ? 1 : 0, U, lim);
  if (e || U % lim->unit_group) return false;
  if (U / lim->unit_group * 32 > lim->max_threads) return false;       // registers
  if (lim->smem == 0 || lim->smem > (uint32_t)kMaxSmemOptin) return false;  // shared memory
  if (cs == 1 && d->Dh > 128) return false;  // heads above 128 units exist only as clusters
  return true;
}

double step_ns(const rnn_desc_t* d, int cs, const FwdLimits& lim) {
  for (const StepRow& r : kStepTable)
    if (r.cell == d->cell && r.Dh == d->Dh && r.ns[log2_cs(cs)] > 0) return r.ns[log2_cs(cs)];
  return model_step_ns(d, cs, lim.unit_group);
}

int device_sms() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

struct PlanChoice {
  int cs, chunk, ctas, waves;
  double us;
};

// L = 1: one layer over T steps; L > 1: the stacked wavefront (chunk_req 0 =
// choose the chunk).  d->cluster != 0 restricts the search to that size.
int plan_search(const rnn_desc_t* d, int L, int sms, int chunk_req, PlanChoice* out) {
  const int nb = (d->B + 7) / 8;
  const int T = d->T > 0 ? d->T : 1;
  bool found = false;
  PlanChoice best{};
  for (int cs : kClusterSizes) {
    if (d->cluster && cs != d->cluster) continue;
    FwdLimits lim;
    if (!cs_limits(d, cs, &lim)) continue;
    const double step = step_ns(d, cs, lim);
    const int ctas = d->NH * nb * cs;
    const int waves = (ctas + sms - 1) / sms;
    const int chunks[6] = {32, 64, 128, 256, 512, T};
    for (int ci = 0; ci < 6; ++ci) {
      int chunk = chunk_req > 0 ? chunk_req : chunks[ci];
      if (L == 1) chunk = T;
      if (chunk > T) chunk = T;
      double us;
      if (L == 1) {
        us = waves * (double)T * step * 1e-3;
      } else {
        // layers resident at once (7/8 of the SMs; the projections take the rest)
        int P = (sms * 7 / 8) / (ctas > 0 ? ctas : 1);
        if (P < 1) P = 1;
        if (P > L) P = L;
        const int nch = (T + chunk - 1) / chunk;
        // the chunk's input projection runs on the SMs the other layers' recurrences leave
        int free_sms = sms - (P - 1) * ctas;
        if (free_sms < 16) free_sms = 16;
        const double dd = (double)d->NH * d->Dh;
        const double proj_us = 2.0 * chunk * d->B * gates_of(d->cell) * dd * dd /
                               (kProjTflops * 1e6 * free_sms / sms);
        const double t_chunk = chunk * step * waves * 1e-3 + proj_us + kChunkOverheadUs;
        const int stages = nch + L - 1 > (L * nch + P - 1) / P ? nch + L - 1 : (L * nch + P - 1) / P;
        us = stages * t_chunk;
      }
      if (!found || us < best.us * 0.995) {
        best = PlanChoice{cs, chunk, ctas, waves, us};
        found = true;
      }
      if (L == 1 || chunk_req > 0) break;
    }
  }
  if (!found) return RNN_ERR_UNSUPPORTED;
  *out = best;
  return RNN_OK;
}

bool bf16_dh_supported(int Dh) {
  return Dh == 32 || Dh == 64 || Dh == 128 || Dh == 256 || Dh == 768;
}

struct Plan {
  bool f32;
  int CS, U, NT, NB, nbslices;
};

int make_plan(const rnn_desc_t* d, Plan* pl) {
  if (d->dtype == RNN_F32) {
    if (d->Dh != 16 && d->Dh != 32 && d->Dh != 64) return RNN_ERR_UNSUPPORTED;
    if (d->cluster > 1) return RNN_ERR_UNSUPPORTED;
    pl->f32 = true;
    pl->CS = 1;
    pl->U = d->Dh;
    pl->NT = 1;
    pl->NB = 8;
  } else {
    if (!bf16_dh_supported(d->Dh)) return RNN_ERR_UNSUPPORTED;
    int cs = d->cluster;
    if (cs == 0) {
      PlanChoice pc;
      if (plan_search(d, 1, device_sms(), 0, &pc) != RNN_OK) return RNN_ERR_UNSUPPORTED;
      cs = pc.cs;
    }
    if (cs != 1 && cs != 2 && cs != 4 && cs != 8 && cs != 16) return RNN_ERR_UNSUPPORTED;
    if (d->Dh % cs) return RNN_ERR_UNSUPPORTED;
    const int U = d->Dh / cs;
    if (U % bf16_unit_group(d->cell)) return RNN_ERR_UNSUPPORTED;
    pl->f32 = false;
    pl->CS = cs;
    pl->U = U;
    pl->NT = 1;
    pl->NB = 8;
  }
  pl->nbslices = (d->B + pl->NB - 1) / pl->NB;
  return RNN_OK;
}

int map_launch_error(int e) {
  if (e == 0) return RNN_OK;
  if (e == -1) return RNN_ERR_NO_CLUSTER;
  if (e == (int)cudaErrorInvalidConfiguration || e == (int)cudaErrorInvalidValue)
    return RNN_ERR_UNSUPPORTED;
  return RNN_ERR_LAUNCH;
}

int launch_forward(const rnn_desc_t* d, const Plan& pl, const FwdParams& p, cudaStream_t s,
                   bool query_only, LaunchInfo* info) {
  if (pl.f32) return launch_fwd_f32(p, d->cell, d->Dh, s, query_only, info);
  switch (d->cell) {
    case RNN_LSTM: return launch_fwd_bf16_lstm(p, d->Dh, pl.NT, s, query_only, info);
    case RNN_GRU: return launch_fwd_bf16_gru(p, d->Dh, pl.NT, s, query_only, info);
    default:
      // hi+lo split of h for the sLSTM while it fits on chip (Dh <= 256)
      return launch_fwd_bf16_slstm(p, d->Dh, pl.NT,
                                   ((d->flags & RNN_FLAG_H_BF16) || d->Dh > 256) ? 0 : 1, s,
                                   query_only, info);
  }
}

FwdParams base_params(const rnn_desc_t* d, const Plan& pl) {
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.T = d->T;
  p.B = d->B;
  p.NH = d->NH;
  p.CS = pl.CS;
  p.U = pl.U;
  p.nbslices = pl.nbslices;
  p.flags = d->flags;
  p.timeout_ns = (d->flags & RNN_FLAG_TEST_TIMEOUT) ? kTestTimeoutNs : kTimeoutNs;
  return p;
}

// Final state <- initial state (or zero) for a zero-length sequence.
int copy_state(float* dst, const float* src, size_t n, cudaStream_t s) {
  if (dst == nullptr) return RNN_OK;
  cudaError_t e = src ? cudaMemcpyAsync(dst, src, n * sizeof(float), cudaMemcpyDeviceToDevice, s)
                      : cudaMemsetAsync(dst, 0, n * sizeof(float), s);
  return e == cudaSuccess ? RNN_OK : RNN_ERR_LAUNCH;
}


// ---------------------------------------------------------------- layer stack --
constexpr int kMaxLayers = 8;
constexpr int kMaxDevices = 64;

// Per-device streams and events of the layer wavefront, created on first use.
struct LayerStreams {
  bool ready = false;
  cudaStream_t s[kMaxLayers];
  cudaEvent_t ev[kMaxLayers], done[kMaxLayers], fork;
};
std::mutex g_stack_mu;
LayerStreams g_streams[kMaxDevices];

int layer_streams(int dev, LayerStreams** out) {
  if (dev < 0 || dev >= kMaxDevices) return RNN_ERR_UNSUPPORTED;
  LayerStreams& ls = g_streams[dev];
  if (!ls.ready) {
    for (int i = 0; i < kMaxLayers; ++i) {
      if (cudaStreamCreateWithFlags(&ls.s[i], cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&ls.ev[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&ls.done[i], cudaEventDisableTiming) != cudaSuccess)
        return RNN_ERR_LAUNCH;
    }
    if (cudaEventCreateWithFlags(&ls.fork, cudaEventDisableTiming) != cudaSuccess)
      return RNN_ERR_LAUNCH;
    ls.ready = true;
  }
  *out = &ls;
  return RNN_OK;
}

int state_arrays(int cell) { return cell == RNN_LSTM ? 2 : (cell == RNN_GRU ? 1 : 4); }

}  // namespace

extern "C" {

const char* rnn_status_str(int status) {
  switch (status) {
    case RNN_OK: return "ok";
    case RNN_ERR_INVALID_ARG: return "invalid argument";
    case RNN_ERR_UNSUPPORTED: return "unsupported shape, dtype or cell";
    case RNN_ERR_MISALIGNED: return "misaligned pointer";
    case RNN_ERR_LAUNCH: return "CUDA launch failed";
    case RNN_ERR_TIMEOUT: return "device wait timed out";
    case RNN_ERR_NO_CLUSTER: return "thread-block cluster cannot be scheduled";
    case RNN_ERR_SCRATCH_LIMIT: return "needs more scratch than the no-allocation entry point holds";
    default: return "unknown status";
  }
}

size_t rnn_stash_size(const rnn_desc_t* d) {
  if (check_desc(d) != RNN_OK) return 0;
  const size_t cells = (size_t)d->T * d->B * d->NH * d->Dh;
  // four gate values + one state (+ the sLSTM normaliser)
  return cells * (d->cell == RNN_SLSTM ? 6 : 5) * sizeof(float);
}

size_t rnn_workspace_size(const rnn_desc_t* d, int pass) {
  if (check_desc(d) != RNN_OK) return 0;
  if (pass == 0) return kStatusBytes;
  // backward: status | bf16(h0) [B,NH,Dh] | bias-gradient partials [slices,NH,G*Dh]
  // fp32 | GRU: recurrent-preactivation gradient bf16 [T,B,NH,3Dh]
  const size_t G = gates_of(d->cell);
  const size_t nb = (size_t)((d->B + 7) / 8);
  size_t o = kStatusBytes;
  o += align_up((size_t)d->B * d->NH * d->Dh * 2, 256);
  o += align_up(nb * d->NH * G * d->Dh * sizeof(float), 256);
  if (d->cell == RNN_GRU) o += align_up((size_t)d->T * d->B * d->NH * G * d->Dh * 2, 256);
  return o;
}

int rnn_fwd_config(const rnn_desc_t* d, int32_t* out6) {
  int st = check_desc(d);
  if (st != RNN_OK) return st;
  if (out6 == nullptr) return RNN_ERR_INVALID_ARG;
  Plan pl;
  if ((st = make_plan(d, &pl)) != RNN_OK) return st;
  LaunchInfo li{};
  FwdParams p = base_params(d, pl);
  int e = launch_forward(d, pl, p, nullptr, true, &li);
  if (e != 0) return map_launch_error(e);
  out6[0] = li.grid;
  out6[1] = li.threads;
  out6[2] = li.cluster;
  out6[3] = li.nb;
  out6[4] = li.smem;
  out6[5] = li.kernel_id;
  return RNN_OK;
}

int rnn_fwd(const rnn_desc_t* d, const void* Wx, const void* R, const float* bias,
            const float* h0, const float* c0, const float* n0, const float* m0, void* h_seq,
            float* hT, float* cT, float* nT, float* mT, void* stash, void* workspace,
            size_t workspace_bytes, void* stream) {
  int st = check_desc(d);
  if (st != RNN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d->B == 0 || d->NH == 0) return RNN_OK;
  Plan pl;
  if ((st = make_plan(d, &pl)) != RNN_OK) return st;
  if (workspace == nullptr || workspace_bytes < rnn_workspace_size(d, 0)) return RNN_ERR_INVALID_ARG;
  const bool train = (d->flags & RNN_FLAG_TRAIN) != 0;
  if (train && d->dtype != RNN_BF16) return RNN_ERR_UNSUPPORTED;
  if (train && stash == nullptr) return RNN_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return RNN_ERR_MISALIGNED;
  const size_t nstate = (size_t)d->B * d->NH * d->Dh;
  if (d->T == 0) {
    int r;
    if ((r = copy_state(hT, h0, nstate, s)) != RNN_OK) return r;
    if (d->cell != RNN_GRU && (r = copy_state(cT, c0, nstate, s)) != RNN_OK) return r;
    if (d->cell == RNN_SLSTM) {
      if ((r = copy_state(nT, n0, nstate, s)) != RNN_OK) return r;
      if ((r = copy_state(mT, m0, nstate, s)) != RNN_OK) return r;
    }
    return RNN_OK;
  }
  if (Wx == nullptr || R == nullptr || h_seq == nullptr) return RNN_ERR_INVALID_ARG;
  if (!aligned(Wx, 16) || !aligned(R, 16) || !aligned(h_seq, 16) || !aligned(stash, 16))
    return RNN_ERR_MISALIGNED;
  const float* fp[] = {bias, h0, c0, n0, m0, hT, cT, nT, mT};
  for (const float* q : fp)
    if (!aligned(q, 4)) return RNN_ERR_MISALIGNED;

  FwdParams p = base_params(d, pl);
  p.Wx = Wx;
  p.R = R;
  p.bias = bias;
  p.h0 = h0;
  p.c0 = c0;
  p.n0 = n0;
  p.m0 = m0;
  p.h_seq = h_seq;
  p.hT = hT;
  p.cT = cT;
  p.nT = nT;
  p.mT = mT;
  if (train) {
    p.stash_gates = static_cast<float*>(stash);
    p.stash_c = p.stash_gates + (size_t)d->T * nstate * 4;
    p.stash_n = p.stash_c + (size_t)d->T * nstate;
  }
  p.status = static_cast<int*>(workspace);
  if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return RNN_ERR_LAUNCH;
  return map_launch_error(launch_forward(d, pl, p, s, false, nullptr));
}

int rnn_input_proj(int32_t M, int32_t N, int32_t K, const void* x, const void* W,
                   const float* bias, void* Wx, void* workspace, size_t workspace_bytes,
                   void* stream) {
  if (M < 0 || N <= 0 || K <= 0) return RNN_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < kStatusBytes) return RNN_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return RNN_ERR_MISALIGNED;
  if (K % 8 != 0 || N % 16 != 0 || M > 65535 * 128) return RNN_ERR_UNSUPPORTED;
  if (M == 0) return RNN_OK;
  if (x == nullptr || W == nullptr || Wx == nullptr) return RNN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(W, 16) || !aligned(Wx, 16) || !aligned(bias, 4))
    return RNN_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return RNN_ERR_LAUNCH;
  return map_launch_error(launch_input_proj_tc(x, W, bias, Wx, M, N, K,
                                               static_cast<int*>(workspace), kTimeoutNs, s));
}

// Stack plan: CTAs per head and time chunk (d->cluster / chunk > 0 are kept).
int stack_plan(const rnn_desc_t* d, int L, int chunk, rnn_desc_t* dl, int* chunk_out) {
  PlanChoice pc;
  if (d->dtype != RNN_BF16 || !bf16_dh_supported(d->Dh)) return RNN_ERR_UNSUPPORTED;
  int st = plan_search(d, L, device_sms(), chunk, &pc);
  if (st != RNN_OK) return st;
  *dl = *d;
  dl->cluster = pc.cs;
  *chunk_out = chunk > 0 ? chunk : pc.chunk;
  return RNN_OK;
}

size_t rnn_stack_workspace_size(const rnn_desc_t* d, int32_t L, int32_t chunk) {
  if (check_desc(d) != RNN_OK || L < 1 || L > kMaxLayers || chunk < 0) return 0;
  if (chunk == 0) {
    rnn_desc_t dl;
    if (stack_plan(d, L, 0, &dl, &chunk) != RNN_OK) return 0;
  }
  const size_t dd = (size_t)d->NH * d->Dh, G = gates_of(d->cell), B = d->B;
  const size_t tc = (size_t)(chunk < d->T ? chunk : (d->T > 0 ? d->T : 1));
  size_t o = kStatusBytes;
  o += align_up((size_t)(L - 1) * d->T * B * dd * 2, 256);              // inner layers' h_seq
  o += (size_t)L * align_up(tc * B * G * dd * 2, 256);                  // Wx of one chunk
  o += (size_t)L * 2 * state_arrays(d->cell) * align_up(B * dd * 4, 256);  // carried states
  return o;
}

int rnn_stack_fwd(const rnn_desc_t* d, int32_t L, int32_t Din, int32_t chunk, const void* x,
                  const void* W_ih0, const void* W_ih, const float* b_ih, const void* R,
                  const float* bias, const float* h0, const float* c0, const float* n0,
                  const float* m0, void* h_seq, float* hT, float* cT, float* nT, float* mT,
                  void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_desc(d);
  if (st != RNN_OK) return st;
  if (L < 1 || L > kMaxLayers || chunk < 0 || Din <= 0) return RNN_ERR_INVALID_ARG;
  if (d->dtype != RNN_BF16 || (d->flags & RNN_FLAG_TRAIN) || Din % 8 != 0)
    return RNN_ERR_UNSUPPORTED;
  if (d->B == 0 || d->NH == 0) return RNN_OK;
  if (workspace == nullptr || workspace_bytes < rnn_stack_workspace_size(d, L, chunk))
    return RNN_ERR_INVALID_ARG;
  rnn_desc_t dplan;
  if ((st = stack_plan(d, L, chunk, &dplan, &chunk)) != RNN_OK) return st;
  d = &dplan;  // the planned CTAs per head
  Plan pl;
  if ((st = make_plan(d, &pl)) != RNN_OK) return st;
  if (!aligned(workspace, 256)) return RNN_ERR_MISALIGNED;
  const float* fp[] = {b_ih, bias, h0, c0, n0, m0, hT, cT, nT, mT};
  for (const float* q : fp)
    if (!aligned(q, 4)) return RNN_ERR_MISALIGNED;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const size_t dd = (size_t)d->NH * d->Dh, G = gates_of(d->cell), B = d->B, T = d->T;
  const size_t nstate = B * dd;
  const int ns = state_arrays(d->cell);
  const float* init[4] = {h0, c0, n0, m0};
  float* fin[4] = {hT, cT, nT, mT};
  auto slot = [&](int k) { return d->cell == RNN_GRU ? (k == 0 ? 0 : -1) : (k < ns ? k : -1); };
  if (T == 0) {
    for (int k = 0; k < 4; ++k)
      if (slot(k) >= 0 && (st = copy_state(fin[k], init[k], (size_t)L * nstate, cs)) != RNN_OK)
        return st;
    return RNN_OK;
  }
  if (x == nullptr || W_ih0 == nullptr || R == nullptr || h_seq == nullptr ||
      (L > 1 && W_ih == nullptr))
    return RNN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(W_ih0, 16) || !aligned(W_ih, 16) || !aligned(R, 16) ||
      !aligned(h_seq, 16))
    return RNN_ERR_MISALIGNED;

  // workspace: status | inner h_seq [L-1][T][B][d] | Wx chunk [L] | states [L][2][ns]
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  size_t o = kStatusBytes;
  __nv_bfloat16* inter = reinterpret_cast<__nv_bfloat16*>(ws + o);
  o += align_up((size_t)(L - 1) * T * B * dd * 2, 256);
  const size_t tcmax = (size_t)(chunk < d->T ? chunk : d->T);
  __nv_bfloat16* wx[kMaxLayers];
  for (int l = 0; l < L; ++l) {
    wx[l] = reinterpret_cast<__nv_bfloat16*>(ws + o);
    o += align_up(tcmax * B * G * dd * 2, 256);
  }
  float* sbuf[kMaxLayers][2][4] = {};
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < 2; ++b)
      for (int k = 0; k < ns; ++k) {
        sbuf[l][b][k] = reinterpret_cast<float*>(ws + o);
        o += align_up(nstate * 4, 256);
      }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RNN_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_stack_mu);
  LayerStreams* ls = nullptr;
  if ((st = layer_streams(dev, &ls)) != RNN_OK) return st;
  if (cudaMemsetAsync(status, 0, sizeof(int), cs) != cudaSuccess ||
      cudaEventRecord(ls->fork, cs) != cudaSuccess)
    return RNN_ERR_LAUNCH;
  for (int l = 0; l < L; ++l)
    if (cudaStreamWaitEvent(ls->s[l], ls->fork, 0) != cudaSuccess) return RNN_ERR_LAUNCH;

  // a layer's projection runs beside the other layers' recurrences: leave them their SMs
  const int rec_ctas = d->NH * pl.nbslices * pl.CS;
  int gemm_cap = sm_count() - (L - 1) * rec_ctas;
  if (gemm_cap < 16) gemm_cap = 16;
  const int nch = (int)((T + chunk - 1) / chunk);
  int err = RNN_OK;
  for (int c = 0; c < nch && err == RNN_OK; ++c) {
    const size_t t0 = (size_t)c * chunk;
    const int tc = (int)(T - t0 < (size_t)chunk ? T - t0 : (size_t)chunk);
    for (int l = 0; l < L && err == RNN_OK; ++l) {
      cudaStream_t s = ls->s[l];
      if (l > 0 && cudaStreamWaitEvent(s, ls->ev[l - 1], 0) != cudaSuccess) {
        err = RNN_ERR_LAUNCH;
        break;
      }
      const __nv_bfloat16* in = l == 0
          ? static_cast<const __nv_bfloat16*>(x) + t0 * B * Din
          : inter + ((size_t)(l - 1) * T + t0) * B * dd;
      const void* W = l == 0 ? W_ih0
                             : static_cast<const void*>(static_cast<const __nv_bfloat16*>(W_ih) +
                                                        (size_t)(l - 1) * G * dd * dd);
      int e = launch_input_proj_tc(in, W, b_ih ? b_ih + (size_t)l * G * dd : nullptr, wx[l],
                                   tc * (int)B, (int)(G * dd), l == 0 ? Din : (int)dd, status,
                                   kTimeoutNs, s, gemm_cap);
      if (e != 0) {
        err = map_launch_error(e);
        break;
      }
      rnn_desc_t dc = *d;
      dc.T = tc;
      FwdParams p = base_params(&dc, pl);
      p.Wx = wx[l];
      p.R = static_cast<const __nv_bfloat16*>(R) + (size_t)l * d->NH * d->Dh * G * d->Dh;
      p.bias = bias ? bias + (size_t)l * d->NH * G * d->Dh : nullptr;
      const float* sin[4];
      for (int k = 0; k < 4; ++k) {
        const int q = slot(k);
        sin[k] = q < 0 ? nullptr
                       : (c == 0 ? (init[k] ? init[k] + (size_t)l * nstate : nullptr)
                                 : sbuf[l][(c - 1) & 1][q]);
      }
      p.h0 = sin[0];
      p.c0 = sin[1];
      p.n0 = sin[2];
      p.m0 = sin[3];
      p.hT = sbuf[l][c & 1][0];
      p.cT = slot(1) >= 0 ? sbuf[l][c & 1][1] : nullptr;
      p.nT = slot(2) >= 0 ? sbuf[l][c & 1][2] : nullptr;
      p.mT = slot(3) >= 0 ? sbuf[l][c & 1][3] : nullptr;
      p.h_seq = l == L - 1 ? static_cast<void*>(static_cast<__nv_bfloat16*>(h_seq) + t0 * B * dd)
                           : static_cast<void*>(inter + ((size_t)l * T + t0) * B * dd);
      p.status = status;
      e = launch_forward(&dc, pl, p, s, false, nullptr);
      if (e != 0 || cudaEventRecord(ls->ev[l], s) != cudaSuccess) {
        err = e != 0 ? map_launch_error(e) : RNN_ERR_LAUNCH;
        break;
      }
    }
  }
  // final states, then the caller's stream waits for every layer (also after an error)
  for (int l = 0; l < L; ++l) {
    cudaStream_t s = ls->s[l];
    if (err == RNN_OK) {
      for (int k = 0; k < 4; ++k) {
        const int q = slot(k);
        if (q < 0 || fin[k] == nullptr) continue;
        if (cudaMemcpyAsync(fin[k] + (size_t)l * nstate, sbuf[l][(nch - 1) & 1][q], nstate * 4,
                            cudaMemcpyDeviceToDevice, s) != cudaSuccess)
          err = RNN_ERR_LAUNCH;
      }
    }
    if (cudaEventRecord(ls->done[l], s) != cudaSuccess ||
        cudaStreamWaitEvent(cs, ls->done[l], 0) != cudaSuccess)
      err = RNN_ERR_LAUNCH;
  }
  return err;
}

// ------------------------------------------------- host-memory forward --
int host_chunk(const rnn_desc_t* d, int chunk) {
  if (chunk > 0) return chunk;
  const int c = (d->T + 3) / 4;  // four chunks: the first copy-in is the only one not hidden
  return c < 64 ? 64 : c;
}

size_t rnn_fwd_host_workspace_size(const rnn_desc_t* d, int32_t chunk) {
  if (check_desc(d) != RNN_OK || chunk < 0) return 0;
  const int tc0 = host_chunk(d, chunk);
  const size_t tc = (size_t)(tc0 < d->T ? tc0 : (d->T > 0 ? d->T : 1));
  const size_t e = d->dtype == RNN_BF16 ? 2 : 4, G = gates_of(d->cell);
  const size_t rows = (size_t)d->B * d->NH;
  size_t o = kStatusBytes;
  o += 2 * align_up(tc * rows * G * d->Dh * e, 256);                      // Wx chunks
  o += 2 * align_up(tc * rows * d->Dh * e, 256);                          // h_seq chunks
  o += 2 * (size_t)state_arrays(d->cell) * align_up(rows * d->Dh * 4, 256);  // carried states
  return o;
}

int rnn_fwd_host(const rnn_desc_t* d, int32_t chunk, const void* Wx_host, const void* R,
                 const float* bias, const float* h0, const float* c0, const float* n0,
                 const float* m0, void* h_seq_host, float* hT, float* cT, float* nT, float* mT,
                 void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_desc(d);
  if (st != RNN_OK) return st;
  if (chunk < 0) return RNN_ERR_INVALID_ARG;
  if (d->flags & RNN_FLAG_TRAIN) return RNN_ERR_UNSUPPORTED;
  if (d->B == 0 || d->NH == 0) return RNN_OK;
  Plan pl;
  if ((st = make_plan(d, &pl)) != RNN_OK) return st;
  if (workspace == nullptr || workspace_bytes < rnn_fwd_host_workspace_size(d, chunk))
    return RNN_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return RNN_ERR_MISALIGNED;
  const float* fp[] = {bias, h0, c0, n0, m0, hT, cT, nT, mT};
  for (const float* q : fp)
    if (!aligned(q, 4)) return RNN_ERR_MISALIGNED;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const size_t nstate = (size_t)d->B * d->NH * d->Dh;
  const int ns = state_arrays(d->cell);
  const float* init[4] = {h0, c0, n0, m0};
  float* fin[4] = {hT, cT, nT, mT};
  auto slot = [&](int k) { return k < ns ? k : -1; };
  if (d->T == 0) {
    for (int k = 0; k < 4; ++k)
      if (slot(k) >= 0 && (st = copy_state(fin[k], init[k], nstate, cs)) != RNN_OK) return st;
    return RNN_OK;
  }
  if (Wx_host == nullptr || R == nullptr || h_seq_host == nullptr) return RNN_ERR_INVALID_ARG;
  if (!aligned(R, 16)) return RNN_ERR_MISALIGNED;

  const int tch = host_chunk(d, chunk);
  const size_t e = d->dtype == RNN_BF16 ? 2 : 4, G = gates_of(d->cell);
  const size_t rows = (size_t)d->B * d->NH;
  const size_t wx_step = rows * G * d->Dh * e, h_step = rows * d->Dh * e;
  const size_t tcmax = (size_t)(tch < d->T ? tch : d->T);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  size_t o = kStatusBytes;
  uint8_t* wxb[2];
  uint8_t* hb[2];
  for (int b = 0; b < 2; ++b) {
    wxb[b] = ws + o;
    o += align_up(tcmax * wx_step, 256);
  }
  for (int b = 0; b < 2; ++b) {
    hb[b] = ws + o;
    o += align_up(tcmax * h_step, 256);
  }
  float* sbuf[2][4] = {};
  for (int b = 0; b < 2; ++b)
    for (int k = 0; k < ns; ++k) {
      sbuf[b][k] = reinterpret_cast<float*>(ws + o);
      o += align_up(nstate * 4, 256);
    }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RNN_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_stack_mu);
  LayerStreams* ls = nullptr;
  if ((st = layer_streams(dev, &ls)) != RNN_OK) return st;
  // copy-in on stream 0, copy-out on stream 1; the recurrence on the caller's stream.
  // events: ev[b] = chunk copied in, ev[2 + b] = chunk computed, ev[4 + b] = chunk copied out
  cudaStream_t sin = ls->s[0], sout = ls->s[1];
  if (cudaMemsetAsync(status, 0, sizeof(int), cs) != cudaSuccess ||
      cudaEventRecord(ls->fork, cs) != cudaSuccess ||
      cudaStreamWaitEvent(sin, ls->fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(sout, ls->fork, 0) != cudaSuccess)
    return RNN_ERR_LAUNCH;
  const int nch = (d->T + tch - 1) / tch;
  int err = RNN_OK;
  for (int c = 0; c < nch && err == RNN_OK; ++c) {
    const int b = c & 1;
    const size_t t0 = (size_t)c * tch;
    const int tc = (int)((size_t)d->T - t0 < (size_t)tch ? (size_t)d->T - t0 : (size_t)tch);
    // in: Wx of chunk c once chunk c-2 no longer reads the buffer
    if ((c >= 2 && cudaStreamWaitEvent(sin, ls->ev[2 + b], 0) != cudaSuccess) ||
        cudaMemcpyAsync(wxb[b], static_cast<const uint8_t*>(Wx_host) + t0 * wx_step,
                        (size_t)tc * wx_step, cudaMemcpyHostToDevice, sin) != cudaSuccess ||
        cudaEventRecord(ls->ev[b], sin) != cudaSuccess) {
      err = RNN_ERR_LAUNCH;
      break;
    }
    // compute: the recurrence over chunk c, from chunk c-1's final state
    if (cudaStreamWaitEvent(cs, ls->ev[b], 0) != cudaSuccess ||
        (c >= 2 && cudaStreamWaitEvent(cs, ls->ev[4 + b], 0) != cudaSuccess)) {
      err = RNN_ERR_LAUNCH;
      break;
    }
    rnn_desc_t dc = *d;
    dc.T = tc;
    FwdParams p = base_params(&dc, pl);
    p.Wx = wxb[b];
    p.R = R;
    p.bias = bias;
    const float* sin_st[4];
    float* sout_st[4];
    for (int k = 0; k < 4; ++k) {
      const int q = slot(k);
      sin_st[k] = q < 0 ? nullptr : (c == 0 ? init[k] : sbuf[(c - 1) & 1][q]);
      sout_st[k] = q < 0 ? nullptr : (c == nch - 1 ? fin[k] : sbuf[c & 1][q]);
    }
    p.h0 = sin_st[0];
    p.c0 = d->cell == RNN_GRU ? nullptr : sin_st[1];
    p.n0 = sin_st[2];
    p.m0 = sin_st[3];
    p.hT = sout_st[0];
    p.cT = d->cell == RNN_GRU ? nullptr : sout_st[1];
    p.nT = sout_st[2];
    p.mT = sout_st[3];
    p.h_seq = hb[b];
    p.status = status;
    const int le = launch_forward(&dc, pl, p, cs, false, nullptr);
    if (le != 0 || cudaEventRecord(ls->ev[2 + b], cs) != cudaSuccess) {
      err = le != 0 ? map_launch_error(le) : RNN_ERR_LAUNCH;
      break;
    }
    // out: h_seq of chunk c
    if (cudaStreamWaitEvent(sout, ls->ev[2 + b], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint8_t*>(h_seq_host) + t0 * h_step, hb[b], (size_t)tc * h_step,
                        cudaMemcpyDeviceToHost, sout) != cudaSuccess ||
        cudaEventRecord(ls->ev[4 + b], sout) != cudaSuccess) {
      err = RNN_ERR_LAUNCH;
      break;
    }
  }
  // the caller's stream waits for both copy streams (also after an error)
  if (cudaEventRecord(ls->done[0], sin) != cudaSuccess ||
      cudaEventRecord(ls->done[1], sout) != cudaSuccess ||
      cudaStreamWaitEvent(cs, ls->done[0], 0) != cudaSuccess ||
      cudaStreamWaitEvent(cs, ls->done[1], 0) != cudaSuccess)
    err = RNN_ERR_LAUNCH;
  return err;
}

int rnn_plan(const rnn_desc_t* d, int32_t L, int32_t sms, int32_t* out5) {
  int st = check_desc(d);
  if (st != RNN_OK) return st;
  if (out5 == nullptr || L < 1 || L > kMaxLayers) return RNN_ERR_INVALID_ARG;
  if (d->dtype != RNN_BF16 || !bf16_dh_supported(d->Dh)) return RNN_ERR_UNSUPPORTED;
  PlanChoice pc;
  if ((st = plan_search(d, L, sms > 0 ? sms : device_sms(), 0, &pc)) != RNN_OK) return st;
  out5[0] = pc.cs;
  out5[1] = pc.chunk;
  out5[2] = pc.ctas;
  out5[3] = pc.waves;
  out5[4] = (int32_t)(pc.us + 0.5);
  return RNN_OK;
}

int rnn_read_status(const void* workspace, void* stream, int* device_status) {
  if (workspace == nullptr || device_status == nullptr) return RNN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return RNN_ERR_LAUNCH;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RNN_ERR_LAUNCH;
  *device_status = (v & kStatusTimeout) ? RNN_ERR_TIMEOUT : RNN_OK;
  return RNN_OK;
}

int rnn_sync_floor(const rnn_desc_t* d, int iters, void* workspace, size_t workspace_bytes,
                   void* stream) {
  int st = check_desc(d);
  if (st != RNN_OK) return st;
  if (iters < 0 || workspace == nullptr || workspace_bytes < kStatusBytes) return RNN_ERR_INVALID_ARG;
  if (d->B == 0 || d->NH == 0 || iters == 0) return RNN_OK;
  Plan pl;
  if ((st = make_plan(d, &pl)) != RNN_OK) return st;
  LaunchInfo li{};
  FwdParams p = base_params(d, pl);
  int e = launch_forward(d, pl, p, nullptr, true, &li);
  if (e != 0) return map_launch_error(e);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return RNN_ERR_LAUNCH;
  return map_launch_error(launch_sync_floor(li, iters, static_cast<int*>(workspace), s));
}

int rnn_bwd(const rnn_desc_t* d, const void* R, const float* h0, const float* c0,
            const float* n0, const void* h_seq, const void* stash, const void* dh_seq,
            const float* dhT, const float* dcT, const float* dnT, void* dWx, float* dR, float* db,
            float* dh0, float* dc0, float* dn0, void* workspace, size_t workspace_bytes,
            void* stream) {
  int st = check_desc(d);
  if (st != RNN_OK) return st;
  if (d->dtype != RNN_BF16) return RNN_ERR_UNSUPPORTED;
  const int Dh = d->Dh;
  if (Dh != 32 && Dh != 64 && Dh != 128 && Dh != 256 && Dh != 768) return RNN_ERR_UNSUPPORTED;
  if (d->B == 0 || d->NH == 0) return RNN_OK;
  if (workspace == nullptr || workspace_bytes < rnn_workspace_size(d, 1)) return RNN_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return RNN_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int G = gates_of(d->cell);
  const size_t nstate = (size_t)d->B * d->NH * Dh;
  const size_t nw = (size_t)d->NH * G * Dh;
  const bool has_c = d->cell != RNN_GRU, has_n = d->cell == RNN_SLSTM;
  if (d->T == 0) {  // no steps: gradients pass straight through to the initial states
    int r;
    if ((r = copy_state(dh0, dhT, nstate, s)) != RNN_OK) return r;
    if (has_c && (r = copy_state(dc0, dcT, nstate, s)) != RNN_OK) return r;
    if (has_n && (r = copy_state(dn0, dnT, nstate, s)) != RNN_OK) return r;
    if (dR && cudaMemsetAsync(dR, 0, nw * Dh * sizeof(float), s) != cudaSuccess) return RNN_ERR_LAUNCH;
    if (db && cudaMemsetAsync(db, 0, nw * sizeof(float), s) != cudaSuccess) return RNN_ERR_LAUNCH;
    return RNN_OK;
  }
  if (R == nullptr || h_seq == nullptr || stash == nullptr || dh_seq == nullptr || dWx == nullptr)
    return RNN_ERR_INVALID_ARG;
  if (!aligned(R, 16) || !aligned(h_seq, 16) || !aligned(stash, 16) || !aligned(dh_seq, 16) ||
      !aligned(dWx, 16))
    return RNN_ERR_MISALIGNED;
  const float* fp[] = {h0, c0, n0, dhT, dcT, dnT, dR, db, dh0, dc0, dn0};
  for (const float* q : fp)
    if (!aligned(q, 8)) return RNN_ERR_MISALIGNED;

  const int nbslices = (d->B + 7) / 8;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  size_t o = kStatusBytes;
  void* h0b = ws + o;
  o += align_up(nstate * 2, 256);
  float* db_part = reinterpret_cast<float*>(ws + o);
  o += align_up((size_t)nbslices * nw * sizeof(float), 256);
  void* drec = d->cell == RNN_GRU ? ws + o : nullptr;

  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.R = R;
  p.dh_seq = dh_seq;
  p.dhT = dhT;
  p.dcT = has_c ? dcT : nullptr;
  p.dnT = has_n ? dnT : nullptr;
  p.stash_gates = static_cast<const float*>(stash);
  p.stash_c = p.stash_gates + (size_t)d->T * nstate * 4;
  p.stash_n = p.stash_c + (size_t)d->T * nstate;
  p.h_init = h0;
  p.c_init = has_c ? c0 : nullptr;
  p.n_init = has_n ? n0 : nullptr;
  p.dWx = dWx;
  p.drec = drec;
  p.dh0 = dh0;
  p.dc0 = has_c ? dc0 : nullptr;
  p.dn0 = has_n ? dn0 : nullptr;
  p.db_part = db ? db_part : nullptr;
  p.status = static_cast<int*>(workspace);
  p.T = d->T;
  p.B = d->B;
  p.NH = d->NH;
  p.nbslices = nbslices;
  p.flags = d->flags;
  p.timeout_ns = (d->flags & RNN_FLAG_TEST_TIMEOUT) ? kTestTimeoutNs : kTimeoutNs;

  if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return RNN_ERR_LAUNCH;
  int e = launch_bwd_bf16(p, d->cell, Dh, s, false, nullptr);
  if (e != 0) return map_launch_error(e);
  if (dR) {
    e = launch_h0_to_bf16(h0, h0b, (int)nstate, s);
    if (e != 0) return map_launch_error(e);
    e = launch_dR_tc(h_seq, h0b, drec ? drec : dWx, dR, d->T, d->B, d->NH, Dh, G, p.status,
                     p.timeout_ns, s);
    if (e != 0) return map_launch_error(e);
  }
  if (db) {
    e = launch_db_reduce(db_part, db, nbslices, (int)nw, s);
    if (e != 0) return map_launch_error(e);
  }
  return RNN_OK;
}

}  // extern "C"
