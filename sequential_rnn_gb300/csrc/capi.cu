// C ABI of the head-wise RNN recurrence (declared in include/rnn.h): the
// single-call entry points -- argument checks, workspace layouts, launches on
// the caller's stream.  The library allocates no device memory.  The launch
// plan lives in plan.cu, the multi-launch runtimes in runtime.cu.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "api.h"

using namespace srnn;
using namespace srnn::api;

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
    case RNN_ERR_BOUNDS: return "an index fell outside its buffer (bounds-check build)";
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
  if (d->B == 0 || d->NH == 0) return clear_status(workspace, workspace_bytes, s);
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
    if ((r = clear_status(workspace, workspace_bytes, s)) != RNN_OK) return r;
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
  if (M == 0) return clear_status(workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
  if (x == nullptr || W == nullptr || Wx == nullptr) return RNN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(W, 16) || !aligned(Wx, 16) || !aligned(bias, 4))
    return RNN_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return RNN_ERR_LAUNCH;
  return map_launch_error(launch_input_proj_tc(x, W, bias, Wx, M, N, K,
                                               static_cast<int*>(workspace), kTimeoutNs, s));
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
  *device_status =
      (v & kStatusTimeout) ? RNN_ERR_TIMEOUT : ((v & kStatusBounds) ? RNN_ERR_BOUNDS : RNN_OK);
  return RNN_OK;
}

int rnn_sync_floor(const rnn_desc_t* d, int iters, void* workspace, size_t workspace_bytes,
                   void* stream) {
  int st = check_desc(d);
  if (st != RNN_OK) return st;
  if (iters < 0 || workspace == nullptr || workspace_bytes < kStatusBytes) return RNN_ERR_INVALID_ARG;
  if (d->B == 0 || d->NH == 0 || iters == 0)
    return clear_status(workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
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
  if (d->B == 0 || d->NH == 0)
    return clear_status(workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
  if (workspace == nullptr || workspace_bytes < rnn_workspace_size(d, 1)) return RNN_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return RNN_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int G = gates_of(d->cell);
  const size_t nstate = (size_t)d->B * d->NH * Dh;
  const size_t nw = (size_t)d->NH * G * Dh;
  const bool has_c = d->cell != RNN_GRU, has_n = d->cell == RNN_SLSTM;
  if (d->T == 0) {  // no steps: gradients pass straight through to the initial states
    int r;
    if ((r = clear_status(workspace, workspace_bytes, s)) != RNN_OK) return r;
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
