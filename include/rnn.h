/*
 * sequential_rnn_gb300 -- C ABI of the head-wise RNN recurrence on GB300 (sm_103a).
 *
 * What is computed (FlashRNN pages: "FlashRNN: I/O-Aware Optimization of
 * Traditional RNNs on modern hardware", abstract -- LSTM, GRU and sLSTM
 * processed as many small heads; blog page "re-examining RNNs from a GPU
 * programming perspective", register-caching and head-wise paragraphs -- the
 * recurrent matrix R stays on chip across the time loop, heads form a
 * block-diagonal R and map to separate thread blocks):
 *
 *   for each head h, batch row b, step t = 0..T-1:
 *     pre_t = Wx[t,b,h,:] + h_{t-1}[b,h,:] @ R[h] + bias[h]        (row vectors)
 *     cell update (below) -> h_t, c_t (, n_t, m_t)
 *
 *   LSTM  gates (i,f,z,o): i,f,o = sigmoid, z = tanh; c = f*c + i*z; h = o*tanh(c)
 *   GRU   gates (r,z,n):   rec = h_{t-1}@R + bias; r = sigm(Wx_r+rec_r);
 *                          z = sigm(Wx_z+rec_z); n = tanh(Wx_n + r*rec_n);
 *                          h = (1-z)*n + z*h_{t-1}
 *   sLSTM gates (i,f,z,o): m_t = max(f~+m, i~); i = exp(i~-m_t); f = exp(f~+m-m_t);
 *                          c = f*c + i*tanh(z~); n = f*n + i; h = sigm(o~)*c/n
 *
 * Layouts (all row-major, contiguous; G = 4 for LSTM/sLSTM, 3 for GRU):
 *   Wx     [T, B, NH, G*Dh]  input dtype     gate-major: column g*Dh + j = gate g, unit j
 *   R      [NH, Dh, G*Dh]    input dtype
 *   bias   [NH, G*Dh]        fp32            (NULL = zeros)
 *   h0,c0,n0,m0 [B, NH, Dh]  fp32            (NULL = zeros; c0 unused by GRU, n0/m0 sLSTM only)
 *   h_seq  [T, B, NH, Dh]    input dtype     h_t for every step (bf16: rounded to nearest even)
 *   hT,cT,nT,mT [B, NH, Dh]  fp32            final states (NULL = not written)
 *
 * Numerics: RNN_F32 computes in fp32 throughout (fp32 FMA contraction,
 * accurate exp/tanh).  RNN_BF16 feeds bf16(h_{t-1}) and bf16 R to the tensor
 * cores with fp32 accumulation; gate math and all states are fp32 (LSTM/GRU
 * gates on the hardware tanh).  For the sLSTM, whose exponential gating
 * amplifies per-step rounding of h by ~10^3 over 4096 steps, h_{t-1} enters
 * the tensor cores as a bf16 pair hi + lo (hi = bf16(h), lo = bf16(h - hi),
 * both products accumulated in fp32; with B <= 4 the two halves share one
 * MMA tile) and tanh(z~) is evaluated as 1 - 2/(e^{2z~}+1) on the
 * 2-ulp exponential instead of the ~2^-11 hardware tanh, for Dh <= 256
 * (Dh = 768 runs the plain bf16 operand: the pair does not fit on chip beside
 * R); RNN_FLAG_H_BF16 turns this off.  With the plain operand the deviation
 * from the exact recurrence grows about linearly with T (~1.5e-5 per step on
 * R ~ U(+-1/sqrt(768)) inputs, fp64 emulation), so an sLSTM with Dh = 768 and
 * T > 768 is rejected with RNN_ERR_UNSUPPORTED unless RNN_FLAG_H_BF16 is set
 * (the caller accepts the plain operand's drift).
 *
 * Ownership: the caller allocates and owns every buffer (device memory),
 * including the workspace and the training stash.  Nothing is allocated by
 * the library.  All calls are asynchronous on `stream` (a cudaStream_t,
 * NULL = legacy default stream).  Host-side checks fail fast with a status
 * and launch nothing.  Device-side failures (a bounded wait that ran out) are
 * recorded in the status word at the start of the workspace; read it with
 * rnn_read_status().  Every call that returns RNN_OK with a workspace leaves
 * its own status there -- 0 also for a call that launches nothing (B, NH or
 * T zero) -- so the workspace needs no clearing by the caller.
 */
#ifndef SEQUENTIAL_RNN_GB300_RNN_H
#define SEQUENTIAL_RNN_GB300_RNN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { RNN_LSTM = 0, RNN_GRU = 1, RNN_SLSTM = 2 } rnn_cell_t;
typedef enum { RNN_F32 = 0, RNN_BF16 = 1 } rnn_dtype_t;

/* desc.flags */
enum {
  RNN_FLAG_TRAIN = 1,              /* forward also writes the stash rnn_bwd needs */
  RNN_FLAG_H_BF16 = 2,             /* sLSTM: plain bf16 h operand and fast gate math
                                      (default for sLSTM is the hi+lo split, see Numerics) */
  RNN_FLAG_TEST_TIMEOUT = 1 << 30  /* test only: the kernel waits on a barrier that nothing
                                      completes, gives up after ~50 ms and reports
                                      RNN_ERR_TIMEOUT in the status word */
};

typedef struct {
  int32_t cell;    /* rnn_cell_t */
  int32_t dtype;   /* rnn_dtype_t: type of Wx, R, h_seq, dh_seq, dWx */
  int32_t T, B, NH, Dh;
  int32_t flags;   /* RNN_FLAG_* */
  int32_t cluster; /* 0 = automatic; else CTAs per head for bf16 (1,2,4,8,16) */
} rnn_desc_t;

typedef enum {
  RNN_OK = 0,
  RNN_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum, small workspace */
  RNN_ERR_UNSUPPORTED = 2, /* shape/dtype/cell combination without a kernel */
  RNN_ERR_MISALIGNED = 3,  /* a pointer violates the alignment stated below */
  RNN_ERR_LAUNCH = 4,      /* the CUDA launch itself failed */
  RNN_ERR_TIMEOUT = 5,     /* device status: a bounded wait ran out, outputs invalid */
  RNN_ERR_NO_CLUSTER = 6,  /* the device cannot co-schedule the needed thread-block cluster */
  RNN_ERR_SCRATCH_LIMIT = 7, /* rnn_fwd_noalloc: the call needs more scratch than its array holds */
  RNN_ERR_BOUNDS = 8         /* device status, bounds-check builds only (libsrnn_bc.so, compiled with
                                -DRNN_BOUNDS_CHECK): a kernel index fell outside its buffer; the
                                access was skipped, outputs invalid */
} rnn_status_t;

/* Bytes of device workspace rnn_fwd (pass 0) / rnn_bwd (pass 1) need.
 * Always >= 256 (the status word lives at offset 0).  0 on invalid desc. */
size_t rnn_workspace_size(const rnn_desc_t* desc, int pass);

/* Bytes of the training stash rnn_fwd writes with RNN_FLAG_TRAIN (bf16 only):
 * four gate values fp32 [T,B,NH,4*Dh], then one state fp32 [T,B,NH,Dh] (LSTM c_t,
 * GRU h_t), then for the sLSTM n_t [T,B,NH,Dh].  Opaque to the caller; pass the
 * same buffer to rnn_bwd. */
size_t rnn_stash_size(const rnn_desc_t* desc);

/* Forward recurrence.  Alignment: Wx, R, h_seq, stash 16 bytes; fp32
 * pointers 4 bytes.  Supported: RNN_F32 with Dh in {16,32,64};
 * RNN_BF16 with Dh in {32,64,128,256,768} (Dh > 128 runs as a thread-block
 * cluster per head).  T == 0 copies the initial states to the final ones;
 * B == 0 or NH == 0 is a no-op.  Returns rnn_status_t. */
int rnn_fwd(const rnn_desc_t* desc, const void* Wx, const void* R, const float* bias,
            const float* h0, const float* c0, const float* n0, const float* m0, void* h_seq,
            float* hT, float* cT, float* nT, float* mT, void* stash, void* workspace,
            size_t workspace_bytes, void* stream);

/* Backward through time (RNN_BF16; LSTM, GRU or sLSTM; Dh in {32,64,128,256,768}),
 * from the stash of a RNN_FLAG_TRAIN forward with the same desc, inputs and
 * h_seq.  Gradients of L = sum(h_seq*dh_seq) + sum(hT*dhT) + sum(cT*dcT) + sum(nT*dnT):
 *   dWx [T,B,NH,G*Dh] input dtype,
 *   dR [NH,Dh,G*Dh] fp32 = sum_t h_{t-1}^T dG_t (h_{-1} = h0 as bf16; dG the
 *      gradient of the recurrent preactivation h@R+b, = dWx except the GRU n block),
 *   db [NH,G*Dh] fp32 = sum_t dG_t, dh0, dc0, dn0 [B,NH,Dh] fp32
 *   (dc0: LSTM/sLSTM, dn0: sLSTM; each of dR/db/dh0/dc0/dn0 may be NULL).
 * h0, c0, n0: the forward's initial states (NULL = zeros).  dhT, dcT, dnT: upstream
 * gradients of the final states (NULL = zero).  The sLSTM stabiliser m is held at
 * its forward values and carries no gradient: exact for any loss of h (h does not
 * depend on m); the dcT, dnT terms are differentiated with m_T held fixed, so
 * that the backward of consecutive time chunks, each fed the next chunk's
 * dh0/dc0/dn0 as dhT/dcT/dnT, composes to the whole sequence's.  dh_seq: input dtype.  Alignment:
 * R, h_seq, dh_seq, dWx, stash 16 bytes; fp32 pointers 8 bytes; workspace 256.
 * The reverse recurrence runs as one thread-block cluster per head slice (as the
 * forward), then the dR contraction (tcgen05 tensor cores) and the db reduction. */
int rnn_bwd(const rnn_desc_t* desc, const void* R, const float* h0, const float* c0,
            const float* n0, const void* h_seq, const void* stash, const void* dh_seq,
            const float* dhT, const float* dcT, const float* dnT, void* dWx, float* dR, float* db,
            float* dh0, float* dc0, float* dn0, void* workspace, size_t workspace_bytes,
            void* stream);

/* rnn_fwd for a sequence in (pinned) host memory: Wx_host [T, B, NH, G*Dh] is
 * read from and h_seq_host [T, B, NH, Dh] written to host memory while the
 * recurrence runs.  Time is cut into chunks of `chunk` steps (0 = automatic:
 * T/8, at least 64 -- or, for bf16 runs that consume Wx at under ~64 GB/s by
 * the plan's step time and pinned, mapped host buffers, the RNN_HOST_DIRECT
 * mode below); chunk c's Wx is copied in on a copy stream while chunk
 * c-1 runs, and chunk c-1's h_seq is copied out on another, so only the first
 * chunk's upload and the last chunk's download are not hidden behind the
 * recurrence.  Each chunk continues from the previous chunk's final state,
 * which gives results identical to one rnn_fwd over all T steps.  R, bias,
 * the initial and final states and the workspace are device memory (as for
 * rnn_fwd); no RNN_FLAG_TRAIN.  The copy streams and events are created on a
 * device's first call and kept (host resources); the enqueue is serialised
 * across host threads; `stream` waits for all of it.  Alignment: R 16 bytes,
 * fp32 pointers 4, workspace 256 and >= rnn_fwd_host_workspace_size() bytes
 * (status word at offset 0, then two Wx chunks, two h_seq chunks and the
 * carried states).  Host memory that is not pinned still works, without the
 * overlap.
 *
 * chunk = RNN_HOST_DIRECT: no staging copies; one rnn_fwd whose kernel reads
 * Wx_host and writes h_seq_host through their device mapping (page-locked host
 * memory on a unified-addressing system, reached over the CPU-GPU link; on
 * Grace-Blackwell NVLink-C2C).  Both buffers must be page-locked and mapped
 * (cudaHostAlloc / cudaMallocHost, or cudaHostRegister with mapping), else
 * RNN_ERR_INVALID_ARG; alignment as for rnn_fwd (16 bytes); workspace as for
 * rnn_fwd. */
#define RNN_HOST_DIRECT (-1)
size_t rnn_fwd_host_workspace_size(const rnn_desc_t* desc, int32_t chunk);
int rnn_fwd_host(const rnn_desc_t* desc, int32_t chunk, const void* Wx_host, const void* R,
                 const float* bias, const float* h0, const float* c0, const float* n0,
                 const float* m0, void* h_seq_host, float* hT, float* cT, float* nT, float* mT,
                 void* workspace, size_t workspace_bytes, void* stream);

/* Input projection, the dense step in front of the recurrence (FlashRNN blog
 * page, register-caching paragraph: only the recurrent weight R has to stay on
 * chip through the sequential time loop; the input weight is applied to all
 * steps at once):
 *   Wx[m, n] = sum_k x[m, k] * W[n, k] + bias[n]
 * x [M, K] bf16 (M = T*B rows of the input sequence), W [N, K] bf16 (rows are
 * output features, as in a linear layer's weight), bias [N] fp32 (NULL = none),
 * Wx [M, N] bf16 (fp32 sum rounded to nearest even once).  With N = NH*G*Dh,
 * Wx is rnn_fwd's input.  fp32 accumulation on the tensor cores (tcgen05, TMA).
 * Requires K % 8 == 0, N % 16 == 0, M <= 8388480.  Alignment: x, W, Wx 16 bytes,
 * bias 4 bytes, workspace 256 bytes and >= 256 bytes (status word at offset 0).
 * M == 0 is a no-op.  Returns rnn_status_t. */
int rnn_input_proj(int32_t M, int32_t N, int32_t K, const void* x, const void* W,
                   const float* bias, void* Wx, void* workspace, size_t workspace_bytes,
                   void* stream);

/* Stacked layers run as a wavefront (FlashRNN blog page, paragraph on cuDNN
 * and layer-level parallelism: layer l+1 can work on step t once layer l has
 * produced h_t).  L layers of one cell and head shape (desc: RNN_BF16, no
 * RNN_FLAG_TRAIN); layer 0 reads x, layer l > 0 reads layer l-1's h_seq; per
 * layer Wx = in W^T + b_ih (as rnn_input_proj) feeds the recurrence.  Time is
 * cut into chunks of `chunk` steps: layer l runs chunk c (its input projection,
 * then the recurrence continuing from chunk c-1's final state) once layer l-1
 * has finished chunk c, each layer on its own stream, so up to L layers run at
 * once.  The result equals running the layers one after the other.
 * Layouts (d = NH*Dh; the G*d projection rows are ordered [NH, G*Dh] like Wx):
 *   x [T, B, Din] bf16;  W_ih0 [G*d, Din] bf16;  W_ih [L-1, G*d, d] bf16 (NULL if
 *   L == 1);  b_ih [L, G*d] fp32 (NULL = 0);  R [L, NH, Dh, G*Dh] bf16;
 *   bias [L, NH, G*Dh] fp32 (NULL = 0);  h0, c0, n0, m0 [L, B, NH, Dh] fp32
 *   (NULL = 0);  h_seq [T, B, NH, Dh] bf16 (last layer);  hT, cT, nT, mT
 *   [L, B, NH, Dh] fp32 (NULL = not written).
 * chunk 0 = chosen by the plan search (rnn_plan), as are the CTAs per head when
 * desc->cluster is 0 (so that the layers' recurrences fit the SMs together).
 * Requires 1 <= L <= 8, chunk >= 0, Din % 8 == 0.  Alignment: bf16 arrays 16
 * bytes, fp32 arrays 4, workspace 256 bytes and >= rnn_stack_workspace_size()
 * (status word at offset 0, then the layers' intermediate h_seq, Wx chunks and
 * carried states).  The per-layer streams and events are created on a device's
 * first call and kept (host resources, no device memory); the enqueue is
 * serialised across host threads.  `stream` waits for all of the work. */
size_t rnn_stack_workspace_size(const rnn_desc_t* desc, int32_t L, int32_t chunk);
int rnn_stack_fwd(const rnn_desc_t* desc, int32_t L, int32_t Din, int32_t chunk, const void* x,
                  const void* W_ih0, const void* W_ih, const float* b_ih, const void* R,
                  const float* bias, const float* h0, const float* c0, const float* n0,
                  const float* m0, void* h_seq, float* hT, float* cT, float* nT, float* mT,
                  void* workspace, size_t workspace_bytes, void* stream);

/* The launch plan the library picks when desc->cluster is 0: an integer search
 * over CTAs per head (1, 2, 4, 8, 16) -- and for L > 1 stacked layers the time
 * chunk -- in the spirit of the FlashRNN card's ConstrINT (hardware limits as
 * integer constraints with divisibility).  A candidate must split the head into
 * whole unit groups of a warp, fit the compiled variant's register budget and
 * shared memory, and (clusters) at most 16 CTAs; the cost is the per-step time
 * (measured on GB300 per cell, Dh and CTAs per head; a latency model where not
 * measured) times the waves the CTAs need over `sms` SMs, and for L > 1 the
 * wavefront's stages given how many layers fit on the SMs at once.
 * sms <= 0: the current device's SM count.  out5[0..4] = CTAs per head, time
 * chunk (T for one layer), CTAs per layer, waves, predicted microseconds.
 * RNN_BF16 only.  Host computation (no launch). */
int rnn_plan(const rnn_desc_t* desc, int32_t L, int32_t sms, int32_t* out5);

/* Synchronises `stream`, reads the device status word of `workspace` into
 * *device_status (RNN_OK, RNN_ERR_TIMEOUT, or in bounds-check builds
 * RNN_ERR_BOUNDS; a timeout is reported first).  Returns RNN_OK if the read
 * itself worked, else RNN_ERR_LAUNCH. */
int rnn_read_status(const void* workspace, void* stream, int* device_status);

/* Measurement aid: runs `iters` iterations of only the per-step
 * synchronisation of the rnn_fwd launch `desc` selects (same grid, cluster
 * shape and barrier kind, no loads and no math).  Its time / iters is the
 * sync floor of one step. */
int rnn_sync_floor(const rnn_desc_t* desc, int iters, void* workspace, size_t workspace_bytes,
                   void* stream);

/* Launch geometry rnn_fwd would use: out[0..5] = grid CTAs, threads per CTA,
 * cluster size, batch rows per CTA, dynamic smem bytes, kernel id. */
int rnn_fwd_config(const rnn_desc_t* desc, int32_t* out6);

const char* rnn_status_str(int status);

/* rnn_fwd for callers that cannot allocate device memory.  The FlashRNN pages
 * have no counterpart; this exists for callers such as a serving process that
 * reserved its whole device-memory budget up front, or a latency-critical loop
 * that must not risk an allocation's implicit device synchronisation.  Same
 * arguments and behaviour as rnn_fwd minus the workspace: its scratch (the
 * device status word) lives in a 4096-byte file-scope __device__ array of the
 * library, held by every GPU that loads the library until the process exits.
 * Calls needing more scratch than that return RNN_ERR_SCRATCH_LIMIT.  The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress)
 * and keeps it for the life of the process, so make that first call before any
 * stream capture, and do not call cudaDeviceReset on that device afterwards (the
 * kept address would then be stale).  Every call shares the array and clears
 * the status word it uses.  Because the caller cannot read the array, the
 * call's device status is delivered through `device_status`: NULL (not
 * reported), or an int the caller owns in device memory or page-locked host
 * memory, which receives the status word by a copy ordered on `stream` after
 * the recurrence -- 0 when every bounded wait completed, nonzero when one ran
 * out (RNN_ERR_TIMEOUT: outputs invalid).  Calls that overlap on the GPU race on
 * the array, so a status delivered to one of them may belong to the other.
 * Allocates nothing (no cudaMalloc / cudaFree, no allocating library call). */
int rnn_fwd_noalloc(const rnn_desc_t* desc, const void* Wx, const void* R, const float* bias,
                    const float* h0, const float* c0, const float* n0, const float* m0,
                    void* h_seq, float* hT, float* cT, float* nT, float* mT, void* stash,
                    int* device_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SEQUENTIAL_RNN_GB300_RNN_H */
