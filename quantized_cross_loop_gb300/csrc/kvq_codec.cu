// kvq_codec.cu — encode (base and residual, K and V), tile directory and
// chain reconstruction kernels.
//
// FlashLoop RFC (vllm-rlt issue #156) §3.3: X̂[1] = deq(q(X[1])); delta[r] =
// X[r] - X̂[r-1]; X̂[r] = X̂[r-1] + deq(q(delta[r])); affine INT4 groups of 64,
// FP16 min and scale; K grouped over (compact) token rows per (head, channel),
// V over channels per (row, head); only active tokens store a residual and
// absent ones inherit. INT4 codec PR (vllm-rlt pull #166), review by 0z5a: codes
// from the FP32 scale before the FP16 metadata is rounded; compact-row K
// groups for sparse residuals.
//
// Work decomposition (ours):
//   encode K  one CTA per (64-row compact group, head); thread = channel; the
//             thread walks its 64 rows in order, so min/max is a plain column
//             scan (no shuffles) and matches the scalar definition bit for bit.
//   encode V  one warp per (stored row, head); lane = 4 channels; min/max over
//             the 16 lanes of a 64-channel group by butterfly shuffles with a
//             lowest-index tie-break (identical bits to an in-order scan, incl. ±0).
//   reconstruct  one warp per (token, head); lane = 4 channels.
#include <cstdio>

#include "kvq_internal.cuh"

namespace kvq {

// ---------------------------------------------------------------- encode K

__global__ void __launch_bounds__(kD) encode_k_kernel(EncodeArgs a) {
  const int g = blockIdx.x;  // compact group
  const int h = blockIdx.y;
  const int d = threadIdx.x;
  const int H = a.prev.n_heads;
  const int r0 = g * kG;
  const int len = min(kG, a.n_rows - r0);
  const int depth = a.prev.depth;

  __shared__ int s_tok[kG];
  __shared__ int s_row[KVQ_MAX_LOOPS][kG];
  __shared__ __align__(16) uint8_t s_codes[kG][kRowBytes];

  if (d < len) {
    int t = a.active ? __ldg(a.active + r0 + d) : r0 + d;
    s_tok[d] = t;
    for (int j = 0; j < depth; ++j) s_row[j][d] = row_of(a.prev.loop[j], t);
  }
  __syncthreads();

  float v[kG];
  float mn = 0.0f, mx = 0.0f;
#pragma unroll
  for (int i = 0; i < kG; ++i) {
    if (i < len) {
      int t = s_tok[i];
      float x = bf16_bits_to_f32(__ldg(a.x + ((long long)t * H + h) * kD + d));
      float val;
      if (depth == 0) {
        val = x;
      } else {
        int rows[KVQ_MAX_LOOPS];
        for (int j = 0; j < depth; ++j) rows[j] = s_row[j][i];
        float xh = chain1(a.prev, depth, rows, h, d);
        val = round_bf16(__fsub_rn(x, xh));
      }
      v[i] = val;
      if (i == 0) {
        mn = val;
        mx = val;
      } else {
        if (val < mn) mn = val;
        if (val > mx) mx = val;
      }
    }
  }
  float s32 = 0.0f;
  if (mx != mn) s32 = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
#pragma unroll
  for (int i = 0; i < kG; ++i) {
    int c = (i < len) ? quantize(v[i], mn, s32) : 0;
    int hi = __shfl_down_sync(0xffffffffu, c, 1);
    if ((d & 1) == 0 && i < len) s_codes[i][d >> 1] = uint8_t(c | (hi << 4));
  }
  long long pi = ((long long)h * ((a.n_rows + kG - 1) / kG) + g) * kD + d;
  a.mins[pi] = f32_to_f16_bits(mn);
  a.scales[pi] = f32_to_f16_bits(s32);
  __syncthreads();
  // len rows x 64 bytes, contiguous in the head-major plane: 16-byte stores.
  uint4* dst = reinterpret_cast<uint4*>(a.codes + ((long long)h * a.n_rows + r0) * kRowBytes);
  const uint4* src = reinterpret_cast<const uint4*>(&s_codes[0][0]);
  for (int k = d; k < len * (kRowBytes / 16); k += blockDim.x) dst[k] = src[k];
}

// ---------------------------------------------------------------- encode V

__global__ void __launch_bounds__(256) encode_v_kernel(EncodeArgs a) {
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int H = a.prev.n_heads;
  const int depth = a.prev.depth;
  __shared__ int s_row[KVQ_MAX_LOOPS];
  __shared__ int s_tok;
  if (threadIdx.x == 0) s_tok = a.active ? __ldg(a.active + row) : row;
  __syncthreads();
  const int t = s_tok;
  if (threadIdx.x < depth) s_row[threadIdx.x] = row_of(a.prev.loop[threadIdx.x], t);
  __syncthreads();
  int rows[KVQ_MAX_LOOPS];
  for (int j = 0; j < depth; ++j) rows[j] = s_row[j];

  for (int h = threadIdx.x >> 5; h < H; h += blockDim.x >> 5) {
    const int c0 = lane * 4;
    uint2 raw = *reinterpret_cast<const uint2*>(a.x + ((long long)t * H + h) * kD + c0);
    float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u), __uint_as_float(raw.y << 16),
                  __uint_as_float(raw.y & 0xFFFF0000u)};
    float v[4];
    if (depth == 0) {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = x[e];
    } else {
      float xh[4];
      chain4(a.prev, depth, rows, h, c0, xh);
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = round_bf16(__fsub_rn(x[e], xh[e]));
    }
    // In-order scan of the lane's 4 channels, then a butterfly over the 16 lanes
    // of the group keeping the lowest channel index among equal values.
    float mn = v[0], mx = v[0];
    int imn = c0, imx = c0;
#pragma unroll
    for (int e = 1; e < 4; ++e) {
      if (v[e] < mn) { mn = v[e]; imn = c0 + e; }
      if (v[e] > mx) { mx = v[e]; imx = c0 + e; }
    }
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) {
      float omn = __shfl_xor_sync(0xffffffffu, mn, off);
      int oimn = __shfl_xor_sync(0xffffffffu, imn, off);
      float omx = __shfl_xor_sync(0xffffffffu, mx, off);
      int oimx = __shfl_xor_sync(0xffffffffu, imx, off);
      if (omn < mn || (omn == mn && oimn < imn)) { mn = omn; imn = oimn; }
      if (omx > mx || (omx == mx && oimx < imx)) { mx = omx; imx = oimx; }
    }
    float s32 = 0.0f;
    if (mx != mn) s32 = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
    int c[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) c[e] = quantize(v[e], mn, s32);
    uint16_t packed = uint16_t(c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12));
    *reinterpret_cast<uint16_t*>(a.codes + ((long long)h * a.n_rows + row) * kRowBytes + lane * 2) = packed;
    if ((lane & 15) == 0) {
      long long pi = ((long long)h * a.n_rows + row) * (kD / kG) + (lane >> 4);
      a.mins[pi] = f32_to_f16_bits(mn);
      a.scales[pi] = f32_to_f16_bits(s32);
    }
  }
}

// ---------------------------------------------------------------- tile directory

__global__ void tile_dir_kernel(const int32_t* __restrict__ active, int n, int n_tiles, int32_t* __restrict__ dir) {
  int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k > n_tiles) return;
  int key = k * KVQ_TILE;
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (__ldg(active + mid) < key) lo = mid + 1;
    else hi = mid;
  }
  dir[k] = lo;
}

// ---------------------------------------------------------------- reconstruct

__global__ void __launch_bounds__(256) reconstruct_kernel(Chain C, uint16_t* __restrict__ out) {
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int H = C.n_heads;
  __shared__ int s_row[KVQ_MAX_LOOPS];
  if (threadIdx.x < C.depth) s_row[threadIdx.x] = row_of(C.loop[threadIdx.x], t);
  __syncthreads();
  int rows[KVQ_MAX_LOOPS];
  for (int j = 0; j < C.depth; ++j) rows[j] = s_row[j];
  for (int h = threadIdx.x >> 5; h < H; h += blockDim.x >> 5) {
    float v[4];
    chain4(C, C.depth, rows, h, lane * 4, v);
    uint2 o;
    o.x = uint32_t(f32_to_bf16_bits(v[0])) | (uint32_t(f32_to_bf16_bits(v[1])) << 16);
    o.y = uint32_t(f32_to_bf16_bits(v[2])) | (uint32_t(f32_to_bf16_bits(v[3])) << 16);
    *reinterpret_cast<uint2*>(out + ((long long)t * H + h) * kD + lane * 4) = o;
  }
}

// ---------------------------------------------------------------- launchers

cudaError_t launch_encode(const EncodeArgs& a, cudaStream_t stream) {
  if (a.n_rows == 0) return cudaSuccess;
  if (a.kind == KVQ_K) {
    dim3 grid((a.n_rows + kG - 1) / kG, a.prev.n_heads);
    encode_k_kernel<<<grid, kD, 0, stream>>>(a);
  } else {
    int warps = a.prev.n_heads < 8 ? a.prev.n_heads : 8;
    encode_v_kernel<<<a.n_rows, 32 * warps, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_tile_dir(const int32_t* active, int n, int T, int32_t* dir, cudaStream_t stream) {
  int n_tiles = (T + KVQ_TILE - 1) / KVQ_TILE;
  int threads = 256;
  int blocks = (n_tiles + 1 + threads - 1) / threads;
  tile_dir_kernel<<<blocks, threads, 0, stream>>>(active, n, n_tiles, dir);
  return cudaGetLastError();
}

cudaError_t launch_reconstruct(const Chain& C, uint16_t* out, cudaStream_t stream) {
  if (C.n_tokens == 0) return cudaSuccess;
  int warps = C.n_heads < 8 ? C.n_heads : 8;
  reconstruct_kernel<<<C.n_tokens, 32 * warps, 0, stream>>>(C, out);
  return cudaGetLastError();
}

}  // namespace kvq
