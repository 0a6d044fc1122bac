// rnn_fwd_noalloc: the forward recurrence for callers that must not allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run the recurrence: a serving process that reserved its whole
// memory budget up front, a real-time loop where an allocation could stall on a
// device-wide synchronisation, or an embedding runtime that owns every byte of
// device memory through its own pool.  They still provide inputs and outputs,
// but not the small scratch workspace rnn_fwd wants.  This entry point keeps
// that scratch in a file-scope __device__ array instead.
//
// The array is static storage of the library: every GPU that loads the library
// holds it until the process exits, and all calls share it.  A call clears the
// part that must start at zero (the device status word); calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on it.
// Since the caller cannot name the array, a call copies its status word, once
// the recurrence is done, into an int the caller owns (device memory or
// page-locked host memory) when it passes one.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/rnn.h"

namespace {

// Largest scratch the array holds; rnn_fwd needs rnn_workspace_size(desc, 0),
// which is 256 bytes for every supported shape.
constexpr size_t kNoAllocScratchBytes = 4096;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Host code must not hand the symbol itself to a kernel (it is a host-side
// stand-in, not a device address); the device address is looked up once per
// device, with that device current, on the first call made on it.
constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void* g_scratch_ptr[kMaxDevices];
cudaError_t g_setup_err[kMaxDevices];

}  // namespace

extern "C" int rnn_fwd_noalloc(const rnn_desc_t* desc, const void* Wx, const void* R,
                               const float* bias, const float* h0, const float* c0,
                               const float* n0, const float* m0, void* h_seq, float* hT, float* cT,
                               float* nT, float* mT, void* stash, int* device_status,
                               void* stream) {
  if (desc == nullptr) return RNN_ERR_INVALID_ARG;
  const size_t need = rnn_workspace_size(desc, 0);
  // a descriptor rnn_fwd refuses (invalid, or a shape without a kernel): its
  // checks return the status before anything touches the device
  if (need == 0)
    return rnn_fwd(desc, Wx, R, bias, h0, c0, n0, m0, h_seq, hT, cT, nT, mT, stash, nullptr, 0,
                   stream);
  if (need > kNoAllocScratchBytes) return RNN_ERR_SCRATCH_LIMIT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RNN_ERR_LAUNCH;
  std::call_once(g_once[dev], [dev]() {
    void* p = nullptr;
    g_setup_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    g_scratch_ptr[dev] = p;
  });
  if (g_setup_err[dev] != cudaSuccess || g_scratch_ptr[dev] == nullptr) return RNN_ERR_LAUNCH;
  // rnn_fwd clears the status word on every path, launching or not
  const int st = rnn_fwd(desc, Wx, R, bias, h0, c0, n0, m0, h_seq, hT, cT, nT, mT, stash,
                         g_scratch_ptr[dev], kNoAllocScratchBytes, stream);
  if (st != RNN_OK || device_status == nullptr) return st;
  // Stream-ordered copy of the status word (no allocation; cudaMemcpyDefault
  // resolves device or page-locked host memory through unified addressing).
  if (cudaMemcpyAsync(device_status, g_scratch_ptr[dev], sizeof(int), cudaMemcpyDefault,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return RNN_ERR_LAUNCH;
  return RNN_OK;
}
