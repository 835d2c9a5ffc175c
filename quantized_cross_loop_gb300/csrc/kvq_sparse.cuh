// kvq_sparse.cuh — arguments and launchers of the sparse decode attention
// kernels (kvq_sparse.cu).
#pragma once

#include "kvq_attn_common.cuh"

namespace kvq {

struct SparseArgs {
  const kvq_request* reqs;
  int32_t n_requests;
  int32_t H;
  int32_t Hq;
  int32_t g;
  int32_t depth;       // reference depth (selection) or the later loop's depth
  int32_t max_tokens;  // largest n_tokens accepted (the logits rows' stride)
  int32_t n_select;    // keys kept per query head (min with n_tokens)
  const uint16_t* q;   // BF16 [B][Hq][128]
  float scale;         // softmax scale (natural-log units)
  float* logits;       // [B][Hq][max_tokens] (log2 units), reference pass
  int32_t* sel_idx;    // [B][Hq][n_select], ascending, -1 past the count
  float* mass;         // [B][Hq]
  float* c_ref;        // [B][Hq][128]
  const float* o_ref;  // [B][Hq][128], later loop
  float* out;          // [B][Hq][128], later loop
  int32_t* err;        // error word
  // later loop on the tensor-core attention kernel
  uint32_t* sel_mask;   // [B][Hq][mask_words]: bit t set for each selected position t
  int32_t mask_words;   // 2 * ceil(max_tokens / 64): whole 64-token tiles
  const float2* stats;  // [B][Hq] softmax (max, sum) of the masked attention
  int32_t refuse_nvfp4; // the masked attention read no NVFP4 loop: requests holding one were refused
};

// Reference pass after the full attention: logits, selection, m and C_ref.
cudaError_t launch_sparse_select_path(const SparseArgs& a, cudaStream_t stream);
// The selection alone, when the tensor-core attention wrote the logits.
cudaError_t launch_sparse_select(const SparseArgs& a, cudaStream_t stream);
// A later loop: the corrected output from the selected keys.
cudaError_t launch_sparse_attn(const SparseArgs& a, cudaStream_t stream);
// A later loop on the tensor-core kernel: the key masks of the selections
// (before the masked attention), then the correction of its output.
cudaError_t launch_sparse_mask(const SparseArgs& a, cudaStream_t stream);
cudaError_t launch_sparse_epilogue(const SparseArgs& a, cudaStream_t stream);

}  // namespace kvq
