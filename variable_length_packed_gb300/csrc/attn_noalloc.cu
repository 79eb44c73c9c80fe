// attn_noalloc.cu — thd_attn_fwd_noalloc: the attention forward for callers that
// cannot allocate device memory.
//
// thd_attn_fwd needs a small workspace (the tile scheduler's work counter and
// the device status word) that the caller allocates.  Some callers have no way
// to do that: plugins hosted by an engine that owns every device allocation and
// hands the plugin no allocator, pipelines that fix their device-memory budget
// at start-up and forbid allocation afterwards, and latency-critical loops that
// must not call cudaMalloc because it can block on the whole device.  The first
// call on a device looks up the buffer's address (scratch_for_current_device);
// make that call before any stream capture begins.  This entry point takes the workspace from a fixed
// buffer compiled into the library instead, so the caller passes only inputs
// and outputs and the library allocates nothing.
//
// The buffer is a file-scope __device__ array: every GPU that loads the library
// holds one copy of it (kNoAllocScratchBytes bytes) until the process exits.
// All calls on a device share that copy, so two calls that overlap on the GPU
// (e.g. on two streams without ordering between them) race on the work counter
// and produce wrong results; calls on one stream, or otherwise ordered, are fine.
// The counter and status word are cleared on the caller's stream at the start of
// every call (by the same path thd_attn_fwd uses), so the buffer needs no
// initialisation and keeps only the last call's contents.  A pipeline wait that
// gives up sets a bit of the status word (byte 8 of the buffer);
// thd_attn_noalloc_status copies that word to the host.
//
// The buffer's device address is cached per device index for the life of the
// process: do not keep using the entry point across cudaDeviceReset (or any
// other teardown of the device's primary context), which may place the
// library's device code, and so the buffer, elsewhere.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/thd_attn.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 256;   // the stated maximum workspace
constexpr size_t kStatusOffset = 8;            // the status word's byte offset in the workspace
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device, looked up once per
// device.  In host code the array's name is only a host-side handle; the
// kernel must receive the address cudaGetSymbolAddress returns.
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return THD_ERR_CUDA;
  if (dev >= kMaxDevices) return THD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return THD_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return THD_OK;
}

}  // namespace

extern "C" int thd_attn_fwd_noalloc(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                                    const int32_t* cu_seqlens_kv, const int32_t* cu_seqlens_q_padded,
                                    const int32_t* cu_seqlens_kv_padded, const uint8_t* seq_is_causal,
                                    int batch_size, int max_seqlen, float softmax_scale, void* out, float* lse,
                                    int total_tokens, int num_heads_q, int num_heads_kv, int head_dim,
                                    int dtype, void* stream) {
  // the workspace the library needs must fit the fixed buffer
  if (thd_attn_workspace_size() > kNoAllocScratchBytes) return THD_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != THD_OK) return st;
  return thd_attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
                      seq_is_causal, batch_size, max_seqlen, softmax_scale, out, lse, total_tokens, num_heads_q,
                      num_heads_kv, head_dim, dtype, scratch, kNoAllocScratchBytes, stream);
}

extern "C" int thd_attn_noalloc_status(uint32_t* status, void* stream) {
  if (!status) return THD_ERR_ARG;
  void* scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != THD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // ordered after the work already queued on `stream`; the host waits for the copy
  if (cudaMemcpyAsync(status, static_cast<char*>(scratch) + kStatusOffset, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                      s) != cudaSuccess)
    return THD_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? THD_OK : THD_ERR_CUDA;
}
