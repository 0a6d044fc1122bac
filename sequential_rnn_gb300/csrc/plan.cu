// Launch planning of the C-ABI library: descriptor checks, the constraint
// search over CTAs per head (and a stack's time chunk), the variant choice
// and the launch of one forward.
#include <cuda_runtime.h>

#include <cstring>

#include "api.h"

namespace srnn {
namespace api {

namespace {
// ------------------------------------------------------------ plan search --
// The launch plan (CTAs per head; for stacked layers also the time chunk) is an
// integer search in the spirit of the FlashRNN card's ConstrINT (hardware
// limits as integer constraints with divisibility): every candidate must
// divide the head into whole warps' unit groups, fit the compiled variant's
// register budget (threads per CTA) and shared memory; among the feasible ones
// the cost is the per-step time times the waves the CTAs need over the SMs
// (and, for a stack, how many layers' recurrences can be resident at once).
// Per-step times: measured on GB300 (bf16 forward, T = 512, inputs in L2), by
// CTAs per head 1, 2, 4, 8, 16; 0 = not measured -> model below.  `hn`: the
// sLSTM rows for at most 4 batch rows (h's hi and lo halves in one n8 tile).
struct StepRow {
  int cell, Dh, hn;
  float ns[5];
};
const StepRow kStepTable[] = {
    {RNN_LSTM, 32, 0, {307, 384, 374, 0, 0}},       {RNN_LSTM, 64, 0, {396, 406, 391, 406, 0}},
    {RNN_LSTM, 128, 0, {0, 515, 432, 439, 499}},    {RNN_LSTM, 256, 0, {0, 0, 763, 615, 703}},
    {RNN_LSTM, 768, 0, {0, 0, 0, 0, 1940}},         {RNN_GRU, 32, 0, {308, 372, 361, 0, 0}},
    {RNN_GRU, 64, 0, {378, 386, 377, 391, 0}},      {RNN_GRU, 128, 0, {661, 520, 412, 423, 477}},
    {RNN_GRU, 256, 0, {0, 1012, 756, 741, 811}},    {RNN_GRU, 768, 0, {0, 0, 0, 0, 1981}},
    {RNN_SLSTM, 32, 0, {381, 426, 438, 0, 0}},      {RNN_SLSTM, 64, 0, {553, 466, 469, 498, 0}},
    {RNN_SLSTM, 128, 0, {0, 863, 680, 668, 707}},   {RNN_SLSTM, 256, 0, {0, 0, 1404, 1077, 1092}},
    {RNN_SLSTM, 768, 0, {0, 0, 0, 0, 2011}},        {RNN_SLSTM, 32, 1, {386, 445, 439, 0, 0}},
    {RNN_SLSTM, 64, 1, {501, 472, 461, 478, 0}},    {RNN_SLSTM, 128, 1, {0, 586, 495, 505, 555}},
    {RNN_SLSTM, 256, 1, {0, 0, 873, 677, 752}},
};
constexpr int kClusterSizes[5] = {1, 2, 4, 8, 16};
constexpr int kMaxSmemOptin = 232448;       // dynamic shared memory per CTA (sm_103)
constexpr double kChunkOverheadUs = 20.0;   // launch + prologue of one stacked chunk
constexpr double kProjTflops = 600.0;       // input-projection GEMM rate on all SMs (chunk sizes)

int log2_cs(int cs) { return cs == 1 ? 0 : cs == 2 ? 1 : cs == 4 ? 2 : cs == 8 ? 3 : 4; }

}  // namespace

// sLSTM h_{t-1} operand: 0 plain bf16; 1 bf16 hi + lo pair as two MMA operands;
// 2 the pair packed into one n8 tile (batches of at most 4 rows per head).
int hsplit_mode(const rnn_desc_t* d) {
  if (d->cell != RNN_SLSTM || (d->flags & RNN_FLAG_H_BF16) || d->Dh > 256) return 0;
  return d->B <= 4 ? 2 : 1;
}

namespace {

// Fallback model for unmeasured points: sync floor of the launch shape plus a
// fixed latency chain plus tensor-pipe issue (8-cycle mma.sync per sub-partition).
double model_step_ns(const rnn_desc_t* d, int cs, int unit_group) {
  const int G = gates_of(d->cell), U = d->Dh / cs, NW = U / unit_group;
  const int per_warp = (unit_group * G + 15) / 16 * (d->Dh / 16) * (hsplit_mode(d) == 1 ? 2 : 1);
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
  else e = fwd_bf16_slstm_limits(d->Dh, hsplit_mode(d), U, lim);
  if (e || U % lim->unit_group) return false;
  if (U / lim->unit_group * 32 > lim->max_threads) return false;       // registers
  if (lim->smem == 0 || lim->smem > (uint32_t)kMaxSmemOptin) return false;  // shared memory
  if (cs == 1 && d->Dh > 128) return false;  // heads above 128 units exist only as clusters
  return true;
}

double step_ns(const rnn_desc_t* d, int cs, const FwdLimits& lim) {
  const int hn = hsplit_mode(d) == 2 ? 1 : 0;
  for (const StepRow& r : kStepTable)
    if (r.cell == d->cell && r.Dh == d->Dh && r.hn == hn && r.ns[log2_cs(cs)] > 0)
      return r.ns[log2_cs(cs)];
  return model_step_ns(d, cs, lim.unit_group);
}

}  // namespace

double plan_step_ns(const rnn_desc_t* d, int cs) {
  FwdLimits lim;
  if (d->dtype != RNN_BF16 || !bf16_dh_supported(d->Dh) || !cs_limits(d, cs, &lim)) return 0.0;
  return step_ns(d, cs, lim);
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

// L = 1: one layer over T steps; L > 1: the stacked wavefront (chunk_req 0 =
// choose the chunk).  d->cluster != 0 restricts the search to that size.
int plan_search(const rnn_desc_t* d, int L, int sms, int chunk_req, PlanChoice* out) {
  const int nbr = hsplit_mode(d) == 2 ? 4 : 8;  // batch rows per CTA
  const int nb = (d->B + nbr - 1) / nbr;
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

int check_desc(const rnn_desc_t* d) {
  if (d == nullptr) return RNN_ERR_INVALID_ARG;
  if (d->cell < RNN_LSTM || d->cell > RNN_SLSTM) return RNN_ERR_INVALID_ARG;
  if (d->dtype != RNN_F32 && d->dtype != RNN_BF16) return RNN_ERR_INVALID_ARG;
  if (d->T < 0 || d->B < 0 || d->NH < 0 || d->Dh <= 0) return RNN_ERR_INVALID_ARG;
  if (d->cluster < 0) return RNN_ERR_INVALID_ARG;
  // sLSTM heads above 256 units take h as one bf16 operand (the hi + lo pair
  // does not fit on chip); its error grows about linearly with the steps
  // (exponential gating is not contractive), so longer sequences need the
  // caller's explicit RNN_FLAG_H_BF16
  if (d->cell == RNN_SLSTM && d->dtype == RNN_BF16 && d->Dh > 256 &&
      !(d->flags & RNN_FLAG_H_BF16) && d->T > kSlstmPlainMaxT)
    return RNN_ERR_UNSUPPORTED;
  return RNN_OK;
}

bool bf16_dh_supported(int Dh) {
  return Dh == 32 || Dh == 64 || Dh == 128 || Dh == 256 || Dh == 768;
}

int make_plan(const rnn_desc_t* d, Plan* pl) {
  if (d->dtype == RNN_F32) {
    if (d->Dh != 16 && d->Dh != 32 && d->Dh != 64) return RNN_ERR_UNSUPPORTED;
    if (d->cluster > 1) return RNN_ERR_UNSUPPORTED;
    pl->f32 = true;
    pl->CS = 1;
    pl->U = d->Dh;
    pl->NT = 1;
    pl->NB = 1;  // one CTA per (head, batch row)
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
    if (U % bf16_unit_group(d->cell, d->Dh, U)) return RNN_ERR_UNSUPPORTED;
    pl->f32 = false;
    pl->CS = cs;
    pl->U = U;
    pl->NT = 1;
    pl->NB = hsplit_mode(d) == 2 ? 4 : 8;
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
      return launch_fwd_bf16_slstm(p, d->Dh, pl.NT, hsplit_mode(d), s, query_only, info);
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

// Status word of a call that launches nothing <- 0, so that reading it never
// returns a status left in that memory before the call.  No workspace (or
// one too small to hold the word): nothing to clear.
int clear_status(void* workspace, size_t workspace_bytes, cudaStream_t s) {
  if (workspace == nullptr || workspace_bytes < sizeof(int) || !aligned(workspace, 4))
    return RNN_OK;
  return cudaMemsetAsync(workspace, 0, sizeof(int), s) == cudaSuccess ? RNN_OK : RNN_ERR_LAUNCH;
}

// Final state <- initial state (or zero) for a zero-length sequence.
int copy_state(float* dst, const float* src, size_t n, cudaStream_t s) {
  if (dst == nullptr) return RNN_OK;
  cudaError_t e = src ? cudaMemcpyAsync(dst, src, n * sizeof(float), cudaMemcpyDeviceToDevice, s)
                      : cudaMemsetAsync(dst, 0, n * sizeof(float), s);
  return e == cudaSuccess ? RNN_OK : RNN_ERR_LAUNCH;
}


}  // namespace api
}  // namespace srnn
