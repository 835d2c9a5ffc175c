// kvq_attn_common.cuh — work decomposition shared by the decode-attention
// kernels: a device-side plan (tile prefix over requests), a flat balanced
// split of all (request, KV head, 64-token tile) work items over a fixed grid,
// partial (max, sum, acc) slots, and the log-sum-exp combine.
//
// Work order: request b, then KV head h, then logical tile k. Unit u = b*H + h
// owns tiles [prefix[b] + h*nt_b, prefix[b] + (h+1)*nt_b), nt_b = ceil(T_b/64).
// CTA c owns the global tile range [floor(c*W/C), floor((c+1)*W/C)). A CTA that
// covers a whole unit writes its output directly; otherwise it writes a partial
// to slot c + u (distinct for every (c, u) pair because ranges are ordered and
// contiguous), and the combine kernel merges the partials of the unit.
#pragma once

#include <utility>

#include "kvq_internal.cuh"

namespace kvq {

constexpr int kMaxG = 8;                          // query heads per KV head
constexpr int kMmaMaxDepth = 4;                   // loops the tensor-core kernel stages per tile
constexpr int kSlotFloats = kMaxG * (kD + 2);     // m[8], l[8], acc[8][128]

struct AttnArgs {
  const kvq_request* reqs;
  int32_t n_requests;
  int32_t H;
  int32_t Hq;
  int32_t g;
  int32_t depth;
  int32_t n_ctas;
  const uint16_t* q;  // BF16 [B][Hq][128]
  float scale;        // softmax scale (natural-log units)
  float* out;         // FP32 [B][Hq][128]
  int32_t* err;       // error word
  int32_t* flags;     // word after the error word, set by the plan: bit 0 = some request has BF16
                      // segments; bit 1 = some accepted request holds an NVFP4 loop within depth
  int32_t* prefix;    // [B+1] tile prefix
  float* partials;    // slots
  float2* stats;      // [B][Hq] (max in log2 units, sum of exponentials) of the packed part
  int32_t nvfp4;      // the table may hold NVFP4 loops (the tensor-core kernel's NVFP4-reading form)
  int32_t refuse_nvfp4;  // the kernel of this call reads no NVFP4 loop: such requests are refused
  // sparse decode (tensor-core kernel only): bit t of word t / 32 of row (b, query head)
  // says key t is selected; the logits of the other keys are dropped. NULL: every key.
  const uint32_t* sel_mask;
  int32_t mask_words;
  // sparse decode reference pass (tensor-core kernel only): every logit (log2
  // units) of key t < logit_stride to logits[(b * Hq + query head) * logit_stride + t]
  float* logits;
  int32_t logit_stride;
  // tensor-core calls: 1 runs the general kernel (64 + c codes, the NVFP4
  // form when nvfp4 is set); 0 runs the mma.sync kernel of kvq_attn_tc.cu for
  // INT4 calls (sparse-decode masks and logits included), or, when tcgen05 is
  // 1 and the call has neither masks nor logits, the tcgen05 kernel of
  // kvq_attn_tcgen05.cu
  int32_t general;
  int32_t tcgen05;
  // 1: the plan kernel clears the error word and the plan flags before its
  // checks (the call's first launch; no separate memset)
  int32_t clear_err;
  // a call whose table may hold NVFP4 loops launches two kernels and the plan
  // picks one: 1 = this INT4 kernel leaves when flags bit 1 is set; 2 = this
  // NVFP4-reading kernel leaves unless it is set; 0 = the kernel always runs
  int32_t dispatch;
};

// Programmatic dependent launches: a kernel launched with launch_dependent()
// may start while its predecessor in the stream finishes; it calls
// wait_prior_grid() before touching anything the predecessor writes (the wait
// returns once the predecessor grid has completed and its memory is visible;
// it does nothing in a kernel launched the ordinary way).
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... P, typename... A>
inline cudaError_t launch_dependent(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                    A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Workspace layout: [0,16) error word (int32 0) and plan flags (int32 1); then int32 prefix[B+1] (rounded to 16 B);
// then (n_ctas + B*H) partial slots of kSlotFloats floats; then float2
// stats[B*Hq] (the packed part's softmax max and sum, merged with the BF16
// segments afterwards).
__host__ __device__ inline size_t ws_prefix_offset() { return 16; }
__host__ __device__ inline size_t ws_partials_offset(int B) {
  return 16 + ((size_t(B) + 1) * 4 + 15) / 16 * 16;
}
__host__ __device__ inline size_t ws_stats_offset(int B, int H, int n_ctas) {
  return ws_partials_offset(B) + (size_t(n_ctas) + size_t(B) * H) * kSlotFloats * 4;
}
__host__ __device__ inline size_t ws_bytes(int B, int H, int Hq, int n_ctas) {
  return ws_stats_offset(B, H, n_ctas) + (size_t(B) * Hq * 8 + 15) / 16 * 16;
}

__device__ __forceinline__ long long cta_start(int c, long long W, int C) { return (long long)c * W / C; }

// Largest c with cta_start(c) <= x, for 0 <= x < W.
__device__ __forceinline__ int cta_of(long long x, long long W, int C) {
  long long c = ((x + 1) * C + W - 1) / W - 1;
  if (c < 0) c = 0;
  if (c > C - 1) c = C - 1;
  return int(c);
}

// Largest b with prefix[b] <= x (prefix is non-decreasing, prefix[0] = 0).
__device__ __forceinline__ int request_of(const int32_t* prefix, int B, long long x) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int n_tiles_of(int T) { return (T + KVQ_TILE - 1) / KVQ_TILE; }

// BF16 segment fields of a request entry (sink within the packed tokens, at
// most KVQ_MAX_SEGMENT tokens in all, aligned buffers for nonzero counts).
__device__ __forceinline__ bool segments_ok(const kvq_request& r) {
  if (r.n_sink < 0 || r.n_tail < 0 || r.n_sink > r.n_tokens || r.n_sink + r.n_tail > KVQ_MAX_SEGMENT) return false;
  auto aligned = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (r.n_sink > 0 && !(aligned(r.sink_k) && aligned(r.sink_v))) return false;
  if (r.n_tail > 0 && !(aligned(r.tail_k) && aligned(r.tail_v))) return false;
  return true;
}

// A request entry the kernels can read without going out of bounds.
__device__ __forceinline__ bool request_ok(const kvq_request& r, int depth) {
  if (r.n_tokens < 0 || r.n_loops < depth || r.n_loops > KVQ_MAX_LOOPS) return false;
  if (!segments_ok(r)) return false;
  if (r.n_tokens == 0) return true;
  if (r.loop[0].active_idx != nullptr || r.loop[0].n_rows != r.n_tokens) return false;
  for (int j = 0; j < depth; ++j) {
    const kvq_loop_ref& L = r.loop[j];
    if (L.n_rows < 0 || L.n_rows > r.n_tokens) return false;
    if (L.active_idx == nullptr && L.n_rows != r.n_tokens) return false;
    if (L.active_idx != nullptr && L.tile_dir == nullptr) return false;
    if (L.n_rows > 0 && (L.k_codes == nullptr || L.v_codes == nullptr || L.k_mins == nullptr || L.k_scales == nullptr ||
        L.v_mins == nullptr || L.v_scales == nullptr))
      return false;
  }
  return true;
}

// A request this call can attend: a consistent entry, and no NVFP4 loop when
// the call's kernel does not read them.
__device__ __forceinline__ bool holds_nvfp4(const kvq_request& r, int depth) {
  for (int j = 0; j < depth && j < KVQ_MAX_LOOPS; ++j)
    if (r.loop[j].flags & (KVQ_LOOP_K_NVFP4 | KVQ_LOOP_V_NVFP4)) return true;
  return false;
}
__device__ __forceinline__ bool nvfp4_refused(const AttnArgs& a, const kvq_request& r) {
  return a.refuse_nvfp4 && holds_nvfp4(r, a.depth);
}
__device__ __forceinline__ bool attn_request_ok(const AttnArgs& a, const kvq_request& r) {
  return request_ok(r, a.depth) && !nvfp4_refused(a, r);
}

cudaError_t launch_plan(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_combine(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_segments(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_attn_mma(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_attn_tcgen05(const AttnArgs& a, cudaStream_t stream);

// The call runs the tcgen05 INT4 kernel (one CTA of the work split per block,
// where the other tensor-core kernels run two per block).
inline bool runs_tcgen05(const AttnArgs& a, bool mma_algo) {
  return mma_algo && !a.general && a.tcgen05 && !a.nvfp4 && a.sel_mask == nullptr && a.logits == nullptr;
}
int attn_ctas(int algo, int device);

}  // namespace kvq
