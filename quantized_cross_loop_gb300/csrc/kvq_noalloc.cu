// kvq_noalloc.cu — packed-KV decode attention for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc or any allocating library routine:
// code that runs while a CUDA graph is being captured, plugins hosted by a
// serving process that owns every device allocation, or hosts with a custom
// allocator the library cannot reach. kvq_decode_attn_packed needs a caller
// workspace for its split-K partials, tile prefix and error word; this entry
// point uses a file-scope device array instead, so the caller only passes the
// request table, the query and the output.
//
// The array is reserved on every device where this code's module is loaded and
// stays there until the process exits. Its device address is looked up once
// per device (cudaGetSymbolAddress, with that device current) on the first call
// made on that device, so that first call must come before any stream capture;
// the address is kept for the life of the process, so the device must not be
// reset once this entry point has been used. The kernels' error word lives in
// the array too: a request they refuse shows only as NaN output rows.
// All calls share the array and leave the last call's contents in it; calls
// that overlap on the GPU (other streams or threads) race on it and must be
// serialised by the caller.
#include <cstdio>
#include <mutex>

#include "kvq_attn_common.cuh"

static __device__ __align__(256) unsigned char g_attn_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace kvq {
void set_error_message(const char* msg);
}

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device (looked up once per device).
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kvq_status kvq_decode_attn_packed_noalloc(const kvq_request* reqs, int n_requests, int n_heads,
                                                     int n_q_heads, int head_dim, int depth, const uint16_t* q,
                                                     float softmax_scale, float* out, kvq_cuda_stream stream) {
  const size_t need = kvq_decode_attn_workspace_bytes(n_requests, n_heads, n_q_heads, head_dim);
  if (need > KVQ_NOALLOC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "n_requests %d x n_heads %d needs %zu bytes of scratch; the static scratch holds %u bytes", n_requests,
             n_heads, need, (unsigned)KVQ_NOALLOC_SCRATCH_BYTES);
    kvq::set_error_message(msg);
    return KVQ_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
    kvq::set_error_message(msg);
    return KVQ_ERR_CUDA;
  }
  return kvq_decode_attn_packed(reqs, n_requests, n_heads, n_q_heads, head_dim, depth, q, softmax_scale, out, scratch,
                                KVQ_NOALLOC_SCRATCH_BYTES, stream);
}
