// Multi-launch runtimes of the C-ABI library: the stacked layers' wavefront
// (rnn_stack_fwd) and the forward over a sequence in host memory
// (rnn_fwd_host).  Both enqueue on per-device streams and events created on
// first use, serialised across host threads, and make the caller's stream wait
// for all of it.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "api.h"

using namespace srnn;
using namespace srnn::api;

namespace {

constexpr int kMaxDevices = 64;

// Per-device streams and events, created on first use: the layer wavefront
// takes one stream per layer, the host-memory forward streams 0 (copy-in) and
// 1 (copy-out).
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

// Time chunk of the host-memory forward.
// Device address of page-locked host memory mapped into the device's address
// space; RNN_ERR_INVALID_ARG for any other pointer (pageable or device memory).
int host_device_alias(const void* host, void** dev) {
  if (host == nullptr) return RNN_ERR_INVALID_ARG;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();  // clear the (non-sticky) error the query recorded
    return RNN_ERR_INVALID_ARG;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return RNN_ERR_INVALID_ARG;
  *dev = a.devicePointer;
  return RNN_OK;
}

// Wx rate (GB/s) below which the automatic host-memory forward reads the mapped
// host buffers directly.  Measured on GB300 per call, direct vs staged copies:
// sLSTM 4x256 B=4 (51 GB/s of Wx) 2.66 vs 2.83 ms; GRU 6x128 B=8 (95 GB/s)
// 1.00 vs 0.95 ms; LSTM 12x64 B=16 (268 GB/s) 1.20 vs 0.67 ms.
constexpr double kHostDirectMaxGBs = 64.0;

int host_chunk(const rnn_desc_t* d, int chunk) {
  if (chunk > 0) return chunk;
  // eight chunks (at least 64 steps each): only the first copy-in and the last
  // copy-out are not hidden; measured on GB300 end to end, eight beat four by
  // 2-6% (12x64 LSTM T=1024: 0.66 vs 0.70 ms) and 16 lose to launch overheads
  const int c = (d->T + 7) / 8;
  return c < 64 ? 64 : c;
}

}  // namespace

extern "C" {

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
  if (d->B == 0 || d->NH == 0)
    return clear_status(workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
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
    if ((st = clear_status(workspace, workspace_bytes, cs)) != RNN_OK) return st;
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
size_t rnn_fwd_host_workspace_size(const rnn_desc_t* d, int32_t chunk) {
  if (check_desc(d) != RNN_OK || chunk < RNN_HOST_DIRECT) return 0;
  if (chunk == RNN_HOST_DIRECT) return kStatusBytes;  // the forward's status word only
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
  if (chunk < RNN_HOST_DIRECT) return RNN_ERR_INVALID_ARG;
  if (d->flags & RNN_FLAG_TRAIN) return RNN_ERR_UNSUPPORTED;
  if (d->B == 0 || d->NH == 0)
    return clear_status(workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
  if (chunk == RNN_HOST_DIRECT) {
    // one forward whose kernel streams Wx from and stores h_seq to the host
    // buffers through their device mapping; only page-locked, mapped memory
    // (the driver reports a device address for it) is accepted
    void* wx_dev = nullptr;
    void* hs_dev = nullptr;
    if (d->T > 0) {
      if ((st = host_device_alias(Wx_host, &wx_dev)) != RNN_OK ||
          (st = host_device_alias(h_seq_host, &hs_dev)) != RNN_OK)
        return st;
    }
    return rnn_fwd(d, wx_dev, R, bias, h0, c0, n0, m0, hs_dev, hT, cT, nT, mT, nullptr, workspace,
                   workspace_bytes, stream);
  }
  Plan pl;
  if ((st = make_plan(d, &pl)) != RNN_OK) return st;
  if (chunk == 0 && d->T > 0 && !pl.f32) {
    // automatic: stream straight from mapped host memory when the recurrence
    // consumes Wx slowly enough for the kernel's own prefetch over the link
    const double sns = plan_step_ns(d, pl.CS);
    const double wx_gbs = sns > 0.0 ? (double)d->B * d->NH * gates_of(d->cell) * d->Dh * 2 / sns
                                    : 1e9;
    void* wx_dev = nullptr;
    void* hs_dev = nullptr;
    if (wx_gbs < kHostDirectMaxGBs && host_device_alias(Wx_host, &wx_dev) == RNN_OK &&
        host_device_alias(h_seq_host, &hs_dev) == RNN_OK)
      return rnn_fwd(d, wx_dev, R, bias, h0, c0, n0, m0, hs_dev, hT, cT, nT, mT, nullptr,
                     workspace, workspace_bytes, stream);
  }
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
    if ((st = clear_status(workspace, workspace_bytes, cs)) != RNN_OK) return st;
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

}  // extern "C"
