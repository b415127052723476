// Decode attention for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc (or any allocator) at
// the point where they run a decode step: code that runs inside a memory
// budget fixed at start-up, an embedding runtime that forbids allocation
// after initialisation, or a host that owns every device allocation itself and
// hands plug-ins only the tensors they read and write.  kvc_decode_attention
// needs a workspace; this file provides one that is not allocated at call
// time: a fixed-size array in the library's own device memory, reserved when
// the library's module is loaded on a GPU and held by that GPU until the
// process exits.
//
// The entry point does the same work as kvc_decode_attention (it calls it);
// only the workspace comes from here.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kvc.h"

namespace {

static_assert(KVC_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// One shared scratch per device.  Every call uses it and leaves its contents
// behind; calls that overlap on the GPU (two streams, or two host threads)
// race on it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KVC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device.  The array's name in
// host code is only a host-side handle, so the address is looked up once per
// device (with that device current) and cached for the life of the process;
// a device reset invalidates it (the header says so).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kvc_status kvc_decode_attention_noalloc(kvc_cache* cache, int32_t seq_begin, int32_t batch,
                                                   const void* d_q, void* d_out, float sm_scale, int32_t flags,
                                                   void* stream) {
  if (!cache) return KVC_ERR_INVALID_ARG;
  const size_t need = kvc_workspace_bytes(cache, batch);
  if (need == 0) return KVC_ERR_INVALID_ARG;
  if (need > (size_t)KVC_NOALLOC_SCRATCH_BYTES) return KVC_ERR_CAPACITY;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KVC_ERR_CUDA;
  // Nothing in the scratch has to start at zero: every value the attention
  // kernels read from their workspace is written earlier in the same call.
  return kvc_decode_attention(cache, seq_begin, batch, d_q, d_out, sm_scale, flags, scratch,
                              (size_t)KVC_NOALLOC_SCRATCH_BYTES, stream);
}
