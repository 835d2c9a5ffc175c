// kvq_codec.cu — encode (base and residual, K and V), tile directory and
// chain reconstruction kernels, for one request or a batch of requests.
//
// FlashLoop RFC (vllm-rlt issue #156) §3.3: X̂[1] = deq(q(X[1])); delta[r] =
// X[r] - X̂[r-1]; X̂[r] = X̂[r-1] + deq(q(delta[r])); affine INT4 groups of 64,
// FP16 min and scale; K grouped over (compact) token rows per (head, channel),
// V over channels per (row, head); only active tokens store a residual and
// absent ones inherit. INT4 codec PR (vllm-rlt pull #166), review by 0z5a: codes
// from the FP32 scale before the FP16 metadata is rounded; compact-row K
// groups for sparse residuals.
//
// Work decomposition (ours). Every kernel runs over a flat list of work items
// spanning all requests of the call; a fixed grid splits the list into
// contiguous ranges, so consecutive items of a CTA usually share a request
// and its chain descriptor (rebuilt in shared memory only when it changes).
//   encode K     item = (64-row compact group, head); thread = channel; the
//                thread walks the group's rows in order, so min/max is a plain
//                column scan and matches the scalar definition bit for bit.
//   encode V     item = 64 stored rows; warp = (row, head) pair; lane = 4
//                channels; min/max over the 16 lanes of a 64-channel group by
//                butterfly shuffles with a lowest-index tie-break (the same bits
//                as an in-order scan, including the sign of zero).
//   tile dir     item = one directory entry (binary search of the index list).
//   reconstruct  item = 64-token logical tile; a shared-memory map gives each
//                token's stored row in every sparse loop; warp = (token, head).
#include "kvq_internal.cuh"

namespace kvq {

__device__ __forceinline__ const kvq_request& req_at(const CodecArgs& a, int b) {
  return a.reqs ? a.reqs[b] : a.one;
}

// Stored rows of the last 64-token tile of loop L (append mode): [*r0, *r0 + return).
__device__ __forceinline__ int last_tile_rows(const kvq_request& R, const kvq_loop_ref& L, int* r0) {
  const int k = R.n_tokens / KVQ_TILE - 1;
  if (L.active_idx == nullptr) {
    *r0 = k * KVQ_TILE;
    return KVQ_TILE;
  }
  *r0 = L.tile_dir[k];
  return L.tile_dir[k + 1] - L.tile_dir[k];
}

__device__ __forceinline__ int items_of(const CodecArgs& a, const kvq_request& R, int mode) {
  if (R.n_tokens < 0 || R.n_loops > KVQ_MAX_LOOPS) return 0;
  if (a.append) {  // the last tile: one K group per head, or one block of at most 64 stored rows
    if (a.loop >= R.n_loops || R.n_tokens < KVQ_TILE || R.n_tokens % KVQ_TILE) return 0;
    const kvq_loop_ref& L = R.loop[a.loop];
    int r0;
    const int m = last_tile_rows(R, L, &r0);
    if (m <= 0) return 0;
    return mode == kModeEncK ? a.H : (mode == kModeEncV ? 1 : 0);
  }
  switch (mode) {
    case kModeEncK: {  // one item per (K group, head)
      if (a.loop >= R.n_loops) return 0;
      const kvq_loop_ref& L = R.loop[a.loop];
      return a.H * k_groups_of((L.flags & KVQ_LOOP_K_TILE) != 0, L.n_rows, R.n_tokens);
    }
    case kModeEncV:
    case kModeNvAmax:
    case kModeNvEnc: {  // one item per 64 stored rows (all heads)
      if (a.loop >= R.n_loops) return 0;
      int n = R.loop[a.loop].n_rows;
      return (n + kG - 1) / kG;
    }
    case kModeTileDir: {
      if (a.loop >= R.n_loops || R.loop[a.loop].active_idx == nullptr) return 0;
      return (R.n_tokens + KVQ_TILE - 1) / KVQ_TILE + 1;
    }
    case kModeReconK: {  // one item per (64-token tile, head)
      if (a.loop > R.n_loops) return 0;
      return ((R.n_tokens + KVQ_TILE - 1) / KVQ_TILE) * a.H;
    }
    default: {  // kModeRecon
      if (a.loop > R.n_loops) return 0;
      return (R.n_tokens + KVQ_TILE - 1) / KVQ_TILE;
    }
  }
}

// Exclusive prefix of work items over the requests of a batch (one CTA).
__global__ void __launch_bounds__(1024) items_plan_kernel(const __grid_constant__ CodecArgs a, int mode,
                                                          int32_t* prefix) {
  __shared__ long long s_carry;
  __shared__ int s_warp[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if (threadIdx.x == 0) {
    s_carry = 0;
    prefix[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < a.n_requests; base += blockDim.x) {
    int b = base + threadIdx.x;
    int v = (b < a.n_requests && !(a.skip && a.skip[b])) ? items_of(a, req_at(a, b), mode) : 0;
    if (mode == kModeNvAmax && v > 0) {  // the NVFP4 encoder's running max |delta| of this stream starts at 0
      const kvq_loop_ref& L = req_at(a, b).loop[a.loop];
      const bool nv = (L.flags & (a.kind == KVQ_K ? KVQ_LOOP_K_NVFP4 : KVQ_LOOP_V_NVFP4)) != 0;
      float* rec = reinterpret_cast<float*>(a.kind == KVQ_K ? L.k_scales : L.v_scales);
      if (nv && rec != nullptr) rec[1] = 0.0f;  // (an INT4 plane here is left alone; the encoder refuses it)
    }
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    long long incl = s_carry + (warp > 0 ? s_warp[warp - 1] : 0) + x;
    if (incl > 0x7FFFFFFFLL) {
      if (a.err) atomicOr(a.err, 2);
      incl = 0x7FFFFFFFLL;
    }
    if (b < a.n_requests) prefix[b + 1] = int(incl);
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_carry = incl;
    __syncthreads();
  }
}

// Contiguous item range of this CTA and the request owning an item.
struct ItemRange {
  long long begin, end;
};

__device__ __forceinline__ ItemRange cta_items(const int32_t* prefix, int n_requests) {
  const long long W = prefix[n_requests];
  ItemRange r;
  r.begin = (long long)blockIdx.x * W / gridDim.x;
  r.end = (long long)(blockIdx.x + 1) * W / gridDim.x;
  return r;
}

__device__ __forceinline__ int owner_of(const int32_t* prefix, int n_requests, long long x) {
  int lo = 0, hi = n_requests - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Owner of item x for a CTA whose previous item belonged to request `cur` (-1:
// none yet). A CTA's items ascend, so the search starts at `cur` and is
// usually a single comparison. Every thread computes the same value.
__device__ __forceinline__ int owner_next(const int32_t* prefix, int n_requests, long long x, int cur) {
  if (cur >= 0 && x < prefix[cur + 1]) return cur;
  int lo = cur >= 0 ? cur + 1 : 0, hi = n_requests - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// One thread fills the chain of loops 0..n-1 of request R for `kind`.
__device__ void fill_chain(const kvq_request& R, int kind, int n, int H, Chain& C) {
  C.depth = n;
  C.kind = kind;
  C.n_tokens = R.n_tokens;
  C.n_heads = H;
  C.any_nvfp4 = 0;
  for (int j = 0; j < n; ++j) {
    planes_of(R, j, kind, C.loop[j]);
    C.any_nvfp4 |= C.loop[j].fmt == KVQ_FMT_NVFP4;
  }
}

__device__ __forceinline__ const uint16_t* source_of(const CodecArgs& a, int b) {
  return a.reqs ? a.x[b] : a.one_x;
}

// ---------------------------------------------------------------- generic kernels (any depth)
//
// One element (or four) at a time with the scalar helpers of kvq_internal.cuh;
// used for chains deeper than the fast kernels below are instantiated for.

// ---------------------------------------------------------------- encode K (generic)

__global__ void __launch_bounds__(kD) encode_k_generic_kernel(const __grid_constant__ CodecArgs a, const int32_t* prefix_ws) {
  const int32_t* prefix = prefix_ws ? prefix_ws : a.one_prefix;
  const int d = threadIdx.x;
  const int H = a.H;
  const int r = a.loop;  // loop written; loops 0..r-1 form the predecessor chain
  __shared__ Chain C;    // C.loop[0..r-1]: predecessor chain; C.loop[r]: output planes
  __shared__ int s_tok[kG];
  __shared__ int s_row[KVQ_MAX_LOOPS][kG];
  __shared__ __align__(16) uint8_t s_codes[kG][kRowBytes];
  __shared__ int s_b;

  const ItemRange ir = cta_items(prefix, a.n_requests);
  int cur_b = -1;
  for (long long it = ir.begin; it < ir.end; ++it) {
    if (d == 0) s_b = owner_of(prefix, a.n_requests, it);
    __syncthreads();
    const int b = s_b;
    if (b != cur_b) {
      if (d == 0) fill_chain(req_at(a, b), KVQ_K, r + 1, H, C);
      cur_b = b;
    }
    __syncthreads();
    if (C.loop[r].fmt != KVQ_FMT_INT4) {  // an NVFP4 output loop: not this kernel's format
      if (threadIdx.x == 0 && a.err) atomicOr(a.err, 64);
      continue;
    }
    const int local = int(it - prefix[b]);
    const int g = local / H, h = local % H;
    const LoopPlanes& O = C.loop[r];
    const int n = O.n_rows;
    // rows of group g: 64 consecutive stored rows, or those of logical tile g
    int r0 = g * kG, len = min(kG, n - r0);
    if (O.ktile && O.sparse) {
      r0 = __ldg(O.tile_dir + g);
      const int r1 = __ldg(O.tile_dir + g + 1);
      len = r1 - r0;
      if (r0 < 0 || r1 > n || len < 0 || len > kG) {  // inconsistent tile map: leave the group
        if (d == 0 && a.err) atomicOr(a.err, 4);
        r0 = 0;
        len = 0;
      }
    }
    const uint16_t* x = source_of(a, b);

    if (d < len) {
      int t = O.sparse ? __ldg(O.active + r0 + d) : r0 + d;
      s_tok[d] = t;
      for (int j = 0; j < r; ++j) s_row[j][d] = row_of(C.loop[j], t);
    }
    __syncthreads();

    float v[kG];
    float mn = 0.0f, mx = 0.0f;
#pragma unroll
    for (int i = 0; i < kG; ++i) {
      if (i < len) {
        int t = s_tok[i];
        float xv = bf16_bits_to_f32(__ldg(x + ((long long)t * H + h) * kD + d));
        float val = xv;
        if (r > 0) {
          int rows[KVQ_MAX_LOOPS];
          for (int j = 0; j < r; ++j) rows[j] = s_row[j][i];
          val = round_bf16(__fsub_rn(xv, chain1(C, r, rows, t, h, d)));
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
    // (a tile with no stored row keeps +0 min and +0 scale)
    long long pi = ((long long)h * O.kgroups + g) * kD + d;
    const_cast<uint16_t*>(O.mins)[pi] = f32_to_f16_bits(mn);
    const_cast<uint16_t*>(O.scales)[pi] = f32_to_f16_bits(s32);
    __syncthreads();
    // len rows x 64 bytes, contiguous in the head-major plane: 16-byte stores.
    uint4* dst = reinterpret_cast<uint4*>(const_cast<uint8_t*>(O.codes) + ((long long)h * O.stride + r0) * kRowBytes);
    const uint4* src = reinterpret_cast<const uint4*>(&s_codes[0][0]);
    for (int k = d; k < len * (kRowBytes / 16); k += blockDim.x) dst[k] = src[k];
  }
}

// ---------------------------------------------------------------- encode V

constexpr int kEncVThreads = 256;

__global__ void __launch_bounds__(kEncVThreads) encode_v_generic_kernel(const __grid_constant__ CodecArgs a,
                                                                const int32_t* prefix_ws) {
  const int32_t* prefix = prefix_ws ? prefix_ws : a.one_prefix;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kEncVThreads / 32;
  const int H = a.H;
  const int r = a.loop;
  __shared__ Chain C;
  __shared__ int s_tok[kG];
  __shared__ int s_row[KVQ_MAX_LOOPS][kG];
  __shared__ int s_b;

  const ItemRange ir = cta_items(prefix, a.n_requests);
  int cur_b = -1;
  for (long long it = ir.begin; it < ir.end; ++it) {
    if (threadIdx.x == 0) s_b = owner_of(prefix, a.n_requests, it);
    __syncthreads();
    const int b = s_b;
    if (b != cur_b) {
      if (threadIdx.x == 0) fill_chain(req_at(a, b), KVQ_V, r + 1, H, C);
      cur_b = b;
    }
    __syncthreads();
    if (C.loop[r].fmt != KVQ_FMT_INT4) {  // an NVFP4 output loop: not this kernel's format
      if (threadIdx.x == 0 && a.err) atomicOr(a.err, 64);
      continue;
    }
    const LoopPlanes& O = C.loop[r];
    const int n = O.n_rows;
    const int r0 = int(it - prefix[b]) * kG;
    const int len = min(kG, n - r0);
    const uint16_t* x = source_of(a, b);
    if (threadIdx.x < len) {
      int t = O.sparse ? __ldg(O.active + r0 + threadIdx.x) : r0 + threadIdx.x;
      s_tok[threadIdx.x] = t;
      for (int j = 0; j < r; ++j) s_row[j][threadIdx.x] = row_of(C.loop[j], t);
    }
    __syncthreads();

    for (int p = warp; p < len * H; p += kWarps) {
      const int i = p / H, h = p % H;
      const int t = s_tok[i];
      const int c0 = lane * 4;
      uint2 raw = *reinterpret_cast<const uint2*>(x + ((long long)t * H + h) * kD + c0);
      float xv[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u), __uint_as_float(raw.y << 16),
                     __uint_as_float(raw.y & 0xFFFF0000u)};
      float v[4];
      if (r == 0) {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = xv[e];
      } else {
        int rows[KVQ_MAX_LOOPS];
        for (int j = 0; j < r; ++j) rows[j] = s_row[j][i];
        float xh[4];
        chain4(C, r, rows, t, h, c0, xh);
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = round_bf16(__fsub_rn(xv[e], xh[e]));
      }
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
      const long long row = r0 + i;
      *reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(O.codes) + ((long long)h * O.stride + row) * kRowBytes +
                                   lane * 2) = packed;
      if ((lane & 15) == 0) {
        long long pi = ((long long)h * O.stride + row) * (kD / kG) + (lane >> 4);
        const_cast<uint16_t*>(O.mins)[pi] = f32_to_f16_bits(mn);
        const_cast<uint16_t*>(O.scales)[pi] = f32_to_f16_bits(s32);
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- NVFP4 residual encode (any depth)
//
// A residual loop in NVFP4 (INT4 codec PR review by 0z5a: E2M1 elements, one
// E4M3 scale per 16 channels of a (row, head), one FP32 scale per stream). Two
// passes over the stream's residual rows, both with item = 64 stored rows and a
// warp per (row, head), lane = channels 4 lane .. 4 lane + 3 (four lanes form a
// block): pass 1 (kAmax) takes max |delta| of the stream into word 1 of its
// tensor-scale record (zeroed beforehand); pass 2 derives s_t from it, then each
// block's E4M3 scale and the E2M1 codes. The residual is recomputed in pass 2
// rather than stored. IEEE divisions, as the format's definition states them.

template <bool kAmax>
__global__ void __launch_bounds__(kEncVThreads) nvfp4_encode_kernel(const __grid_constant__ CodecArgs a,
                                                                   const int32_t* prefix_ws) {
  const int32_t* prefix = prefix_ws ? prefix_ws : a.one_prefix;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kEncVThreads / 32;
  const int H = a.H;
  const int r = a.loop;
  __shared__ Chain C;
  __shared__ int s_tok[kG];
  __shared__ int s_row[KVQ_MAX_LOOPS][kG];
  __shared__ int s_b;

  const ItemRange ir = cta_items(prefix, a.n_requests);
  int cur_b = -1;
  for (long long it = ir.begin; it < ir.end; ++it) {
    if (threadIdx.x == 0) s_b = owner_of(prefix, a.n_requests, it);
    __syncthreads();
    const int b = s_b;
    if (b != cur_b) {
      if (threadIdx.x == 0) fill_chain(req_at(a, b), a.kind, r + 1, H, C);
      cur_b = b;
    }
    __syncthreads();
    const LoopPlanes& O = C.loop[r];
    if (r < 1 || O.fmt != KVQ_FMT_NVFP4) {  // the table does not hold an NVFP4 residual here
      if (threadIdx.x == 0 && a.err) atomicOr(a.err, 64);
      continue;
    }
    const int n = O.n_rows;
    const int r0 = int(it - prefix[b]) * kG;
    const int len = min(kG, n - r0);
    const uint16_t* x = source_of(a, b);
    if (threadIdx.x < len) {
      int t = O.sparse ? __ldg(O.active + r0 + threadIdx.x) : r0 + threadIdx.x;
      s_tok[threadIdx.x] = t;
      for (int j = 0; j < r; ++j) s_row[j][threadIdx.x] = row_of(C.loop[j], t);
    }
    __syncthreads();
    float* rec = reinterpret_cast<float*>(const_cast<uint16_t*>(O.scales));
    float st = 0.0f, six_st = 0.0f;
    bool all_zero = true;
    if (!kAmax) {
      const float amax = rec[1];
      all_zero = !(amax > 0.0f);
      st = __fdiv_rn(amax, 2688.0f);  // 6 * 448: the largest block scale times the largest E2M1 value
      six_st = __fmul_rn(6.0f, st);
    }
    float tmax = 0.0f;
    for (int p = warp; p < len * H; p += kWarps) {
      const int i = p / H, h = p % H;
      const int t = s_tok[i];
      const int c0 = lane * 4;
      const uint2 raw = *reinterpret_cast<const uint2*>(x + ((long long)t * H + h) * kD + c0);
      const float xv[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                           __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
      int rows[KVQ_MAX_LOOPS];
      for (int j = 0; j < r; ++j) rows[j] = s_row[j][i];
      float xh[4], v[4];
      chain4(C, r, rows, t, h, c0, xh);
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = round_bf16(__fsub_rn(xv[e], xh[e]));
      float ab = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
      if (kAmax) {
        tmax = fmaxf(tmax, ab);
        continue;
      }
      ab = fmaxf(ab, __shfl_xor_sync(0xffffffffu, ab, 1));  // the block's four lanes
      ab = fmaxf(ab, __shfl_xor_sync(0xffffffffu, ab, 2));
      const uint32_t sb = all_zero ? 0u : f32_to_e4m3(__fdiv_rn(ab, six_st));
      const float eb = __fmul_rn(e4m3_to_f32(sb), st);
      uint32_t packed = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) packed |= (eb == 0.0f ? 0u : f32_to_e2m1(__fdiv_rn(v[e], eb))) << (4 * e);
      const long long row = r0 + i;
      *reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(O.codes) + ((long long)h * O.stride + row) * kRowBytes +
                                   lane * 2) = uint16_t(packed);
      if ((lane & 3) == 0)
        reinterpret_cast<uint8_t*>(const_cast<uint16_t*>(O.mins))[((long long)h * O.stride + row) * (kD / 16) + (lane >> 2)] =
            uint8_t(sb);
    }
    if (kAmax) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      if (lane == 0 && tmax > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(rec + 1), __float_as_uint(tmax));
    } else if (r0 == 0 && threadIdx.x == 0) {
      rec[0] = st;  // the stream's tensor scale, once
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- tile directory

__global__ void __launch_bounds__(256) tile_dir_kernel(const __grid_constant__ CodecArgs a, const int32_t* prefix_ws) {
  const int32_t* prefix = prefix_ws ? prefix_ws : a.one_prefix;
  const long long W = prefix[a.n_requests];
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < W; it += (long long)gridDim.x * blockDim.x) {
    const int b = owner_of(prefix, a.n_requests, it);
    const kvq_loop_ref& L = req_at(a, b).loop[a.loop];
    const int k = int(it - prefix[b]);
    const int key = k * KVQ_TILE;
    int lo = 0, hi = L.n_rows;
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      if (__ldg(L.active_idx + mid) < key) lo = mid + 1;
      else hi = mid;
    }
    L.tile_dir[k] = lo;
  }
}

// ---------------------------------------------------------------- reconstruct

constexpr int kReconThreads = 256;

__global__ void __launch_bounds__(kReconThreads) reconstruct_generic_kernel(const __grid_constant__ CodecArgs a,
                                                                    const int32_t* prefix_ws) {
  const int32_t* prefix = prefix_ws ? prefix_ws : a.one_prefix;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kReconThreads / 32;
  const int H = a.H;
  const int depth = a.loop;
  __shared__ Chain C;
  __shared__ int s_map[KVQ_MAX_LOOPS][KVQ_TILE];
  __shared__ int s_b;

  const ItemRange ir = cta_items(prefix, a.n_requests);
  int cur_b = -1;
  for (long long it = ir.begin; it < ir.end; ++it) {
    if (threadIdx.x == 0) s_b = owner_of(prefix, a.n_requests, it);
    __syncthreads();
    const int b = s_b;
    if (b != cur_b) {
      if (threadIdx.x == 0) fill_chain(req_at(a, b), a.kind, depth, H, C);
      cur_b = b;
    }
    __syncthreads();
    const int k = int(it - prefix[b]);
    const int t0 = k * KVQ_TILE;
    const int nvalid = min(KVQ_TILE, C.n_tokens - t0);
    for (int idx = threadIdx.x; idx < depth * KVQ_TILE; idx += blockDim.x) {
      int j = idx / KVQ_TILE, tt = idx % KVQ_TILE;
      s_map[j][tt] = (C.loop[j].sparse || tt >= nvalid) ? -1 : t0 + tt;
    }
    __syncthreads();
    for (int j = 1; j < depth; ++j) {
      const LoopPlanes& L = C.loop[j];
      if (!L.sparse) continue;
      int c0 = __ldg(L.tile_dir + k), c1 = __ldg(L.tile_dir + k + 1);
      if (c0 < 0 || c1 > L.n_rows || c0 > c1 || c1 - c0 > KVQ_TILE) {
        if (threadIdx.x == 0 && a.err) atomicOr(a.err, 4);
        continue;
      }
      for (int c = c0 + threadIdx.x; c < c1; c += blockDim.x) {
        int tt = __ldg(L.active + c) - t0;
        if (tt >= 0 && tt < KVQ_TILE) s_map[j][tt] = c;
        else if (a.err) atomicOr(a.err, 4);
      }
    }
    __syncthreads();
    uint16_t* out = a.reqs ? a.out[b] : a.one_out;
    for (int p = warp; p < nvalid * H; p += kWarps) {
      const int tt = p / H, h = p % H;
      int rows[KVQ_MAX_LOOPS];
      for (int j = 0; j < depth; ++j) rows[j] = s_map[j][tt];
      float v[4];
      chain4(C, depth, rows, t0 + tt, h, lane * 4, v);
      uint2 o;
      o.x = uint32_t(f32_to_bf16_bits(v[0])) | (uint32_t(f32_to_bf16_bits(v[1])) << 16);
      o.y = uint32_t(f32_to_bf16_bits(v[2])) | (uint32_t(f32_to_bf16_bits(v[3])) << 16);
      *reinterpret_cast<uint2*>(out + ((long long)(t0 + tt) * H + h) * kD + lane * 4) = o;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- fast kernels (chains of up to 4 loops)

constexpr int kFastMaxDepth = 4;  // deepest chain the fast kernels are instantiated for
//
// The same arithmetic as the generic kernels, two channels at a time:
//  - decode RN_bf16(min + scale * c) takes one FP32 FMA per channel: scale * c
//    is exact (an FP16 significand times a 4-bit code), so the FMA rounds once
//    exactly where the generic code rounds the sum; the pair is then converted
//    to BF16 in one instruction;
//  - the chain add and the residual subtraction run on BF16 pairs with a single
//    rounding (add.rn.bf16x2 / sub.rn.bf16x2). For BF16 operands that equals
//    rounding the FP32 result to BF16: the exact sum of two BF16 values fits in
//    FP32 unless their exponents differ by more than 15, and then both
//    roundings return the larger operand;
//  - a code is rint(d * RN32(1 / scale)) instead of rint(RN32(d / scale)). The
//    two quotients differ by less than 1.5 ulp of 16 (2.9e-6), so their
//    rounding to an integer agrees unless the product lies within 4e-6 of a
//    half-integer; such elements, and non-finite products, take the IEEE
//    division of the generic path;
//  - min and max come from BF16 pair min/max; when a group's min or max is
//    zero its sign is re-taken from the first zero in scan order, which is the
//    one the in-order scan keeps.
namespace fast {

constexpr float kMagic23 = 8388608.0f;         // 2^23: x + 2^23 rounds x in [0, 2^23) to an integer
constexpr float kTieWindow = 0.5f - 4.0e-6f;  // |y - rint(y)| above this: exact division

__device__ __forceinline__ uint32_t bf2_add(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf2_min(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// {RN_bf16(v.x), RN_bf16(v.y)} with v.x in the low half
__device__ __forceinline__ uint32_t f2_to_bf2(float2 v) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(v.y), "f"(v.x));
  return d;
}
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) { return make_float2(bf_lo(v), bf_hi(v)); }
__device__ __forceinline__ float2 f16x2_to_f2(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}
__device__ __forceinline__ uint32_t f16_pair(float lo, float hi) {
  return uint32_t(f32_to_f16_bits(lo)) | (uint32_t(f32_to_f16_bits(hi)) << 16);
}

// One codes byte (low nibble = even channel) -> the BF16 pair of decodes,
// with the FP32 min m and scale s of each channel.
__device__ __forceinline__ uint32_t dequant_byte(uint32_t byte, float2 m, float2 s) {
  const float2 c = __fadd2_rn(make_float2(__uint_as_float((byte & 0xFu) | 0x4B000000u),
                                          __uint_as_float((byte >> 4) | 0x4B000000u)),
                              make_float2(-kMagic23, -kMagic23));
  return f2_to_bf2(__ffma2_rn(s, c, m));
}

// One codes word (byte k = channels 2k, 2k+1) -> four BF16 pairs, one min and
// scale for all eight channels.
__device__ __forceinline__ void dequant_word(uint32_t w, float2 m, float2 s, uint32_t* out) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 c = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7440 + k)),
                                            __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7440 + k))),
                                make_float2(-kMagic23, -kMagic23));
    out[k] = f2_to_bf2(__ffma2_rn(s, c, m));
  }
}

// One codes word -> four BF16 pairs with the min and scale of each pair.
__device__ __forceinline__ void dequant_word_pp(uint32_t w, const float2* m, const float2* s, uint32_t* out) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 c = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7440 + k)),
                                            __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7440 + k))),
                                make_float2(-kMagic23, -kMagic23));
    out[k] = f2_to_bf2(__ffma2_rn(s[k], c, m[k]));
  }
}

// Codes of a BF16 pair against the FP32 min, scale and RN32(1 / scale) of each
// channel (reciprocal 0 for a constant group): code(lo) | code(hi) << 4.
__device__ __forceinline__ uint32_t quant_pair(uint32_t v, float2 mn, float2 rc, float2 s32) {
  const float2 x = bf2_to_f2(v);
  const float2 y = __fmul2_rn(__fadd2_rn(x, make_float2(-mn.x, -mn.y)), rc);
  const float2 z = __fadd2_rn(y, make_float2(kMagic23, kMagic23));
  const float2 e = __ffma2_rn(__fadd2_rn(z, make_float2(-kMagic23, -kMagic23)), make_float2(-1.0f, -1.0f), y);
  uint32_t code = (__float_as_uint(z.x) & 0xFu) | ((__float_as_uint(z.y) & 0xFu) << 4);
  if (!(fabsf(e.x) <= kTieWindow && fabsf(e.y) <= kTieWindow))
    code = uint32_t(quantize(x.x, mn.x, s32.x)) | (uint32_t(quantize(x.y, mn.y, s32.y)) << 4);
  return code;
}

// quant_pair without the division: the product codes, and in *near bit 0 / 1
// the channels whose product lies too close to a half-integer (or is not
// finite) to decide; the caller gives those quantize() later. Exact ties are
// common on BF16 data (up to ~2% of residual pairs), so a warp that ran the
// IEEE division for every pair one of its lanes flags would take it on a large
// share of its pairs; collecting the flags first lets the lanes that need it
// run it together.
__device__ __forceinline__ uint32_t quant_pair_fast(uint32_t v, float2 mn, float2 rc, uint32_t* near) {
  const float2 x = bf2_to_f2(v);
  const float2 y = __fmul2_rn(__fadd2_rn(x, make_float2(-mn.x, -mn.y)), rc);
  const float2 z = __fadd2_rn(y, make_float2(kMagic23, kMagic23));
  const float2 e = __ffma2_rn(__fadd2_rn(z, make_float2(-kMagic23, -kMagic23)), make_float2(-1.0f, -1.0f), y);
  *near = uint32_t(!(fabsf(e.x) <= kTieWindow)) | (uint32_t(!(fabsf(e.y) <= kTieWindow)) << 1);
  return (__float_as_uint(z.x) & 0xFu) | ((__float_as_uint(z.y) & 0xFu) << 4);
}

__device__ __forceinline__ float scale_of(float mn, float mx) {
  return (mx != mn) ? __fdiv_rn(__fsub_rn(mx, mn), 15.0f) : 0.0f;
}
__device__ __forceinline__ float recip_of(float s32) { return s32 != 0.0f ? __frcp_rn(s32) : 0.0f; }

}  // namespace fast

// ---------------------------------------------------------------- K parameters in shared memory

// A K group's parameters staged as FP32 (min lo, min hi, scale lo, scale hi)
// per channel pair. Pair P is stored in slot kpar_slot(P): the eight lanes of a
// row, each reading pair 8 sub + k in the same instruction, hit eight different
// 16-byte bank groups.
constexpr int kKParGroups = 6;  // groups of one predecessor loop staged per item
__device__ __forceinline__ int kpar_slot(int pair) { return (pair & ~7) | (((pair & 7) + (pair >> 3)) & 7); }

// Stages groups g0 .. g0 + ng - 1 of head h of loop L (K) into par[0 .. ng-1][64].
__device__ __forceinline__ void stage_kpar(const LoopPlanes& L, int h, int g0, int ng, float4 (*par)[kD / 2]) {
  const long long G = L.kgroups;
  for (int idx = threadIdx.x; idx < ng * (kD / 2); idx += blockDim.x) {
    const int gi = idx / (kD / 2), pair = idx % (kD / 2);
    const long long pi = ((long long)h * G + g0 + gi) * kD + 2 * pair;
    const float2 m = fast::f16x2_to_f2(__ldg(reinterpret_cast<const uint32_t*>(L.mins + pi)));
    const float2 s = fast::f16x2_to_f2(__ldg(reinterpret_cast<const uint32_t*>(L.scales + pi)));
    par[gi][kpar_slot(pair)] = make_float4(m.x, m.y, s.x, s.y);
  }
}

// Parameters of the 16 channels 16 sub .. 16 sub + 15 of K group `grp` of
// head h of K loop L: from the staged groups when the group is among them,
// else from the planes.
__device__ __forceinline__ void load_kpar16(const LoopPlanes& L, int h, int grp, int sub,
                                            const float4 (*par)[kD / 2], int g0, int ng, float2* m, float2* s) {
  const int gi = grp - g0;
  if (gi >= 0 && gi < ng) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 q = par[gi][8 * sub + ((k + sub) & 7)];
      m[k] = make_float2(q.x, q.y);
      s[k] = make_float2(q.z, q.w);
    }
  } else {
    const long long pi = ((long long)h * L.kgroups + grp) * kD + 16 * sub;
    const uint4* mp = reinterpret_cast<const uint4*>(L.mins + pi);
    const uint4* sp = reinterpret_cast<const uint4*>(L.scales + pi);
    const uint4 m0 = __ldg(mp), m1 = __ldg(mp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
    const uint32_t mw[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      m[k] = fast::f16x2_to_f2(mw[k]);
      s[k] = fast::f16x2_to_f2(sw[k]);
    }
  }
}

// Decodes the 16 channels 16 sub .. 16 sub + 15 of one stored K row (codes cw,
// K group grp) into 8 BF16 pairs.
__device__ __forceinline__ void dequant16_k(const LoopPlanes& L, int h, int grp, uint2 cw, int sub,
                                            const float4 (*par)[kD / 2], int g0, int ng, uint32_t* out) {
  float2 m[8], s[8];
  load_kpar16(L, h, grp, sub, par, g0, ng, m, s);
  fast::dequant_word_pp(cw.x, m, s, out);
  fast::dequant_word_pp(cw.y, m + 4, s + 4, out + 4);
}

// ---------------------------------------------------------------- encode K (fast)
//
// item = (K group, head), 256 threads, two phases. A K group is 64 consecutive
// stored rows, or (tile grouping of a sparse loop) the stored rows of one
// 64-token logical tile, found through the tile directory.
//  1. Residuals: eight lanes per row (lane `sub` = channels 16 sub .. +15), a
//     warp four rows; every load of a row is issued before its arithmetic and
//     the BF16 residual pairs go to a shared [row][pair] tile.
//  2. Columns: thread (pair p, quarter q) scans rows 16 q .. 16 q + 15 of pair
//     p; the four partial min/max are merged in row order, then each thread
//     quantises its rows into a shared code tile that leaves in 16-byte stores.

constexpr int kEncKThreads = 256;

template <int R>
struct EncKSmem {
  uint32_t delta[kG][kD / 2];                  // residual BF16 pairs
  uint8_t codes[kG][kRowBytes];                // output codes
  float4 par[R > 0 ? R : 1][kKParGroups][kD / 2];  // staged predecessor parameters
  uint32_t pmn[4][kD / 2], pmx[4][kD / 2];     // partial min/max per row quarter
  float4 qp[kD / 2];                           // per pair: min lo, min hi, 1/scale lo, 1/scale hi
  float2 qs[kD / 2];                           // per pair: scales
  Chain C;
  int tok[kG];
  int row[R > 0 ? R : 1][kG];
  int glo[R > 0 ? R : 1], ghi[R > 0 ? R : 1];
};

// Blocks per SM: five for the base, four for residual loops. The barriers
// between the phases leave a block idle, so more resident blocks pay even at the
// price of a few spilled words (measured: four against three, 6-10% faster for
// residual loops; five, slower there, 9% faster for the base).
template <int R>
__global__ void __launch_bounds__(kEncKThreads, R == 0 ? 5 : 4)
    encode_k_fast_kernel(const __grid_constant__ CodecArgs a, const int32_t* prefix_ws) {
  using namespace fast;
  constexpr int kWarps = kEncKThreads / 32;
  const int32_t* prefix = prefix_ws ? prefix_ws : a.one_prefix;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane & 7, lg = lane >> 3;
  const int H = a.H;
  __shared__ EncKSmem<R> S;

  const ItemRange ir = cta_items(prefix, a.n_requests);
  int cur_b = -1;
  for (long long it = ir.begin; it < ir.end; ++it) {
    const int b = owner_next(prefix, a.n_requests, it, cur_b);
    if (b != cur_b) {
      __syncthreads();  // every thread is done with the previous request's chain
      if (tid == 0) fill_chain(req_at(a, b), KVQ_K, R + 1, H, S.C);
      cur_b = b;
    }
    if (tid < R) {
      S.glo[tid] = 0x7FFFFFFF;
      S.ghi[tid] = -1;
    }
    __syncthreads();
    if (S.C.any_nvfp4) {  // NVFP4 loops: the INT4-only fast path refuses the request
      if (tid == 0 && a.err) atomicOr(a.err, 64);
      continue;
    }
    const int local = int(it - prefix[b]);
    // append mode: the item is the last tile's group (the table already counts the tile)
    const int g = a.append ? S.C.n_tokens / kG - 1 : local / H, h = local % H;
    const LoopPlanes& O = S.C.loop[R];
    const int n = O.n_rows;
    int r0 = g * kG, len = min(kG, n - r0);
    if (O.ktile && O.sparse) {
      r0 = __ldg(O.tile_dir + g);
      const int r1 = __ldg(O.tile_dir + g + 1);
      len = r1 - r0;
      if (r0 < 0 || r1 > n || len < 0 || len > kG) {  // inconsistent tile map: leave the group
        if (tid == 0 && a.err) atomicOr(a.err, 4);
        continue;
      }
    }
    const long long opi = ((long long)h * O.kgroups + g) * kD;  // this group's params
    if (len == 0) {  // a logical tile with no stored row: +0 min and +0 scale
      if (tid < kD / 2) {
        *reinterpret_cast<uint32_t*>(const_cast<uint16_t*>(O.mins) + opi + 2 * tid) = 0u;
        *reinterpret_cast<uint32_t*>(const_cast<uint16_t*>(O.scales) + opi + 2 * tid) = 0u;
      }
      continue;
    }
    const uint16_t* x = source_of(a, b);
    if (a.append) x -= (long long)(S.C.n_tokens - KVQ_TILE) * H * kD;  // the tile's source holds its 64 tokens
    if (tid < len) {
      const int t = O.sparse ? __ldg(O.active + r0 + tid) : r0 + tid;
      S.tok[tid] = t;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int row = row_of(S.C.loop[j], t);
        S.row[j][tid] = row;
        if (row >= 0) {
          const int kg = k_group(S.C.loop[j], t, row);
          atomicMin(&S.glo[j], kg);
          atomicMax(&S.ghi[j], kg);
        }
      }
    }
    __syncthreads();
    if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0) {  // batch source not 16-byte aligned: skip
      if (tid == 0 && a.err) atomicOr(a.err, 16);
      continue;
    }
    int g0[R > 0 ? R : 1], ng[R > 0 ? R : 1];
#pragma unroll
    for (int j = 0; j < R; ++j) {
      g0[j] = S.glo[j];
      ng[j] = S.ghi[j] >= g0[j] ? S.ghi[j] - g0[j] + 1 : 0;
      if (ng[j] > kKParGroups) ng[j] = 0;  // too spread: read the planes instead
      stage_kpar(S.C.loop[j], h, g0[j], ng[j], S.par[j]);
    }
    __syncthreads();

    // ---- phase 1: residual rows (both halves unrolled, so that the second
    // half's loads issue early, except with two predecessor loops, where the
    // extra live registers spill and it measured slower)
#pragma unroll(R == 2 ? 1 : 2)
    for (int i0 = 0; i0 < kG; i0 += 4 * kWarps) {
      const int i = i0 + 4 * warp + lg;
      const bool live = i < len;
      uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
      uint2 cw[R > 0 ? R : 1];
      int rows[R > 0 ? R : 1];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        cw[j] = make_uint2(0, 0);
        rows[j] = -1;
      }
      if (live) {
        const int t = S.tok[i];
        const uint4* src = reinterpret_cast<const uint4*>(x + ((long long)t * H + h) * kD + 16 * sub);
        xa = __ldg(src);
        xb = __ldg(src + 1);
#pragma unroll
        for (int j = 0; j < R; ++j) {
          rows[j] = S.row[j][i];
          if (rows[j] >= 0) {
            const LoopPlanes& L = S.C.loop[j];
            cw[j] = __ldg(reinterpret_cast<const uint2*>(L.codes + ((long long)h * L.stride + rows[j]) * kRowBytes +
                                                         8 * sub));
          }
        }
      }
      uint32_t d[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      if (R > 0) {
        uint32_t acc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = 0;
#pragma unroll
        for (int j = 0; j < R; ++j) {
          if (rows[j] < 0) continue;
          uint32_t dq[8];
          dequant16_k(S.C.loop[j], h, k_group(S.C.loop[j], S.tok[i], rows[j]), cw[j], sub, S.par[j], g0[j], ng[j],
                      dq);
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[k] = (j == 0) ? dq[k] : bf2_add(acc[k], dq[k]);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) d[k] = bf2_sub(d[k], acc[k]);
      }
      if (live) {
        uint4* dst = reinterpret_cast<uint4*>(&S.delta[i][8 * sub]);
        dst[0] = make_uint4(d[0], d[1], d[2], d[3]);
        dst[1] = make_uint4(d[4], d[5], d[6], d[7]);
      }
    }
    __syncthreads();

    // ---- phase 2: per channel pair p, rows of quarter q (held in registers)
    const int p = tid & (kD / 2 - 1), q = tid >> 6;
    const int nr = min(16, len - 16 * q);  // rows of this quarter (<= 0: none)
    if (nr > 0) {
      uint32_t v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = S.delta[16 * q + min(k, nr - 1)][p];  // repeats leave min/max unchanged
      uint32_t mn2 = v[0], mx2 = v[0];
#pragma unroll
      for (int k = 1; k < 16; ++k) {
        mn2 = bf2_min(mn2, v[k]);
        mx2 = bf2_max(mx2, v[k]);
      }
      S.pmn[q][p] = mn2;
      S.pmx[q][p] = mx2;
    }
    __syncthreads();
    if (q == 0) {  // the pair's parameters, once
      const int nq = (len + 15) / 16;
      uint32_t mn2 = S.pmn[0][p], mx2 = S.pmx[0][p];
      for (int qq = 1; qq < nq; ++qq) {
        mn2 = bf2_min(mn2, S.pmn[qq][p]);
        mx2 = bf2_max(mx2, S.pmx[qq][p]);
      }
      float mn[2] = {bf_lo(mn2), bf_hi(mn2)}, mx[2] = {bf_lo(mx2), bf_hi(mx2)};
      if (mn[0] == 0.0f || mn[1] == 0.0f || mx[0] == 0.0f || mx[1] == 0.0f) {
        // the in-order scan keeps the first zero it meets: take its sign
        bool done[4] = {mn[0] != 0.0f, mn[1] != 0.0f, mx[0] != 0.0f, mx[1] != 0.0f};
        for (int i = 0; i < len; ++i) {
          const uint32_t w = S.delta[i][p];
          const float lo = bf_lo(w), hi = bf_hi(w);
          if (!done[0] && lo == 0.0f) { mn[0] = lo; done[0] = true; }
          if (!done[2] && lo == 0.0f) { mx[0] = lo; done[2] = true; }
          if (!done[1] && hi == 0.0f) { mn[1] = hi; done[1] = true; }
          if (!done[3] && hi == 0.0f) { mx[1] = hi; done[3] = true; }
        }
      }
      const float s0 = scale_of(mn[0], mx[0]), s1 = scale_of(mn[1], mx[1]);
      S.qp[p] = make_float4(mn[0], mn[1], recip_of(s0), recip_of(s1));
      S.qs[p] = make_float2(s0, s1);
      const long long pi = opi + 2 * p;
      *reinterpret_cast<uint32_t*>(const_cast<uint16_t*>(O.mins) + pi) = f16_pair(mn[0], mn[1]);
      *reinterpret_cast<uint32_t*>(const_cast<uint16_t*>(O.scales) + pi) = f16_pair(s0, s1);
    }
    __syncthreads();
    if (nr > 0) {
      const float4 qp = S.qp[p];
      const float2 mnv = make_float2(qp.x, qp.y), rc = make_float2(qp.z, qp.w), sv = S.qs[p];
      uint32_t pend = 0;  // bit 2k + c: channel c of row k needs the division
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (k < nr) {
          uint32_t nb;
          S.codes[16 * q + k][p] = uint8_t(quant_pair_fast(S.delta[16 * q + k][p], mnv, rc, &nb));
          pend |= nb << (2 * k);
        }
      while (pend) {  // the flagged channels (this thread's rows only: no warp-wide work needed)
        const int bit = __ffs(pend) - 1;
        pend &= pend - 1;
        const int k = bit >> 1, c = bit & 1;
        const uint32_t w = S.delta[16 * q + k][p];
        const uint32_t code = uint32_t(c ? quantize(bf_hi(w), mnv.y, sv.y) : quantize(bf_lo(w), mnv.x, sv.x));
        uint8_t& byte = S.codes[16 * q + k][p];
        byte = uint8_t((byte & ~(0xFu << (4 * c))) | (code << (4 * c)));
      }
    }
    __syncthreads();
    // len rows x 64 bytes, contiguous in the head-major plane
    if (tid < len * (kRowBytes / 16)) {
      uint4* dst = reinterpret_cast<uint4*>(const_cast<uint8_t*>(O.codes) + ((long long)h * O.stride + r0) * kRowBytes);
      dst[tid] = reinterpret_cast<const uint4*>(&S.codes[0][0])[tid];
    }
  }
}

// ---------------------------------------------------------------- encode V (fast)
//
// item = 64 stored rows (all heads). Eight lanes cover one (row, head): lane
// `sub` holds channels 16 sub .. 16 sub + 15, four lanes one V group; a warp
// takes four consecutive rows of one head, so the codes (4 x 64 B), the
// parameters (4 x 4 B) and each source row (256 B) are contiguous. Every load
// of a (row, head) is issued before its arithmetic.

constexpr int kEncVFastThreads = 256;

template <int R>
__global__ void __launch_bounds__(kEncVFastThreads, 5) encode_v_fast_kernel(const __grid_constant__ CodecArgs a,
                                                                         const int32_t* prefix_ws) {
  using namespace fast;
  constexpr int RA = R > 0 ? R : 1;
  constexpr int kWarps = kEncVFastThreads / 32;
  const int32_t* prefix = prefix_ws ? prefix_ws : a.one_prefix;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane & 7, lg = lane >> 3;
  const int H = a.H;
  __shared__ Chain C;
  __shared__ int s_tok[kG];
  __shared__ int s_row[RA][kG];

  const ItemRange ir = cta_items(prefix, a.n_requests);
  int cur_b = -1;
  for (long long it = ir.begin; it < ir.end; ++it) {
    const int b = owner_next(prefix, a.n_requests, it, cur_b);
    if (b != cur_b) {
      __syncthreads();  // every thread is done with the previous request's chain
      if (threadIdx.x == 0) fill_chain(req_at(a, b), KVQ_V, R + 1, H, C);
      cur_b = b;
    }
    __syncthreads();
    if (C.any_nvfp4) {  // NVFP4 loops: the INT4-only fast path refuses the request
      if (threadIdx.x == 0 && a.err) atomicOr(a.err, 64);
      continue;
    }
    const LoopPlanes& O = C.loop[R];
    const int n = O.n_rows;
    int r0 = int(it - prefix[b]) * kG, len = min(kG, n - r0);
    const uint16_t* x = source_of(a, b);
    if (a.append) {  // the stored rows of the last tile (the table already counts it)
      const int k = C.n_tokens / KVQ_TILE - 1;
      r0 = O.sparse ? __ldg(O.tile_dir + k) : k * KVQ_TILE;
      len = O.sparse ? __ldg(O.tile_dir + k + 1) - r0 : KVQ_TILE;
      if (r0 < 0 || len < 0 || len > kG || r0 + len > n) len = 0;
      x -= (long long)(C.n_tokens - KVQ_TILE) * H * kD;  // the tile's source holds its 64 tokens
    }
    if (threadIdx.x < len) {
      const int t = O.sparse ? __ldg(O.active + r0 + threadIdx.x) : r0 + threadIdx.x;
      s_tok[threadIdx.x] = t;
#pragma unroll
      for (int j = 0; j < R; ++j) s_row[j][threadIdx.x] = row_of(C.loop[j], t);
    }
    __syncthreads();
    if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0) {
      if (threadIdx.x == 0 && a.err) atomicOr(a.err, 16);
      continue;
    }
    const int nquads = H * (kG / 4);
    for (int qd = warp; qd < nquads; qd += kWarps) {
      const int h = qd / (kG / 4);
      const int i = (qd % (kG / 4)) * 4 + lg;
      const bool live = i < len;
      uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
      uint2 cw[RA];
      uint32_t m16[RA], s16[RA];
      bool have[RA];
#pragma unroll
      for (int j = 0; j < RA; ++j) {
        cw[j] = make_uint2(0, 0);
        m16[j] = s16[j] = 0;
        have[j] = false;
      }
      if (live) {
        const int t = s_tok[i];
        const uint4* src = reinterpret_cast<const uint4*>(x + ((long long)t * H + h) * kD + 16 * sub);
        xa = __ldg(src);
        xb = __ldg(src + 1);
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const int row = s_row[j][i];
          if (row >= 0) {
            const LoopPlanes& L = C.loop[j];
            const long long rr = (long long)h * L.stride + row;
            cw[j] = __ldg(reinterpret_cast<const uint2*>(L.codes + rr * kRowBytes + 8 * sub));
            m16[j] = __ldg(L.mins + rr * (kD / kG) + (sub >> 2));
            s16[j] = __ldg(L.scales + rr * (kD / kG) + (sub >> 2));
            have[j] = true;
          }
        }
      }
      uint32_t d[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      if (R > 0) {
        uint32_t acc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = 0;
#pragma unroll
        for (int j = 0; j < R; ++j) {
          if (!have[j]) continue;
          const float mf = f16_bits_to_f32(uint16_t(m16[j])), sf = f16_bits_to_f32(uint16_t(s16[j]));
          uint32_t dq[8];
          dequant_word(cw[j].x, make_float2(mf, mf), make_float2(sf, sf), dq);
          dequant_word(cw[j].y, make_float2(mf, mf), make_float2(sf, sf), dq + 4);
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[k] = (j == 0) ? dq[k] : bf2_add(acc[k], dq[k]);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) d[k] = bf2_sub(d[k], acc[k]);
      }
      const uint32_t m2 = bf2_min(bf2_min(bf2_min(d[0], d[1]), bf2_min(d[2], d[3])),
                                  bf2_min(bf2_min(d[4], d[5]), bf2_min(d[6], d[7])));
      const uint32_t M2 = bf2_max(bf2_max(bf2_max(d[0], d[1]), bf2_max(d[2], d[3])),
                                  bf2_max(bf2_max(d[4], d[5]), bf2_max(d[6], d[7])));
      float mn = fminf(bf_lo(m2), bf_hi(m2)), mx = fmaxf(bf_lo(M2), bf_hi(M2));
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {  // the four lanes of this V group
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      }
      if (__any_sync(0xffffffffu, live && (mn == 0.0f || mx == 0.0f))) {
        // the first zero of the group in channel order carries the sign the scan keeps
        bool has = false;
        float fz = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float lo = bf_lo(d[k]), hi = bf_hi(d[k]);
          if (!has && lo == 0.0f) { has = true; fz = lo; }
          if (!has && hi == 0.0f) { has = true; fz = hi; }
        }
        const unsigned ball = __ballot_sync(0xffffffffu, has);
        const unsigned grp = ball & (0xFu << (lane & ~3));
        const float first = __shfl_sync(0xffffffffu, fz, grp ? __ffs(grp) - 1 : lane);
        if (mn == 0.0f) mn = first;
        if (mx == 0.0f) mx = first;
      }
      const float s32 = scale_of(mn, mx);
      const float2 mnv = make_float2(mn, mn), sv = make_float2(s32, s32);
      const float rcs = recip_of(s32);
      const float2 rc = make_float2(rcs, rcs);
      uint32_t w0 = 0, w1 = 0, pend = 0;  // pend bit 2k + c: channel c of pair k needs the division
      if (R == 0) {  // base data: ties are rare (~0.2% of elements), the per-pair fallback is cheaper
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          w0 |= quant_pair(d[k], mnv, rc, sv) << (8 * k);
          w1 |= quant_pair(d[4 + k], mnv, rc, sv) << (8 * k);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t n0, n1;
          w0 |= quant_pair_fast(d[k], mnv, rc, &n0) << (8 * k);
          w1 |= quant_pair_fast(d[4 + k], mnv, rc, &n1) << (8 * k);
          pend |= (n0 << (2 * k)) | (n1 << (2 * (4 + k)));
        }
      }
      while (R > 0 && __any_sync(0xffffffffu, pend != 0)) {  // the flagged channels, one per lane per round
        if (pend) {
          const int bit = __ffs(pend) - 1;
          pend &= pend - 1;
          const int k = bit >> 1, c = bit & 1;
          uint32_t dv = d[0];
#pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            if (k == kk) dv = d[kk];
          const uint32_t code = uint32_t(quantize(c ? bf_hi(dv) : bf_lo(dv), mn, s32));
          const int sh = 8 * (k & 3) + 4 * c;
          if (k < 4) w0 = (w0 & ~(0xFu << sh)) | (code << sh);
          else w1 = (w1 & ~(0xFu << sh)) | (code << sh);
        }
      }
      const uint32_t mp = f32_to_f16_bits(mn), sp = f32_to_f16_bits(s32);
      const uint32_t mp1 = __shfl_down_sync(0xffffffffu, mp, 4), sp1 = __shfl_down_sync(0xffffffffu, sp, 4);
      if (live) {
        const long long rr = (long long)h * O.stride + r0 + i;
        *reinterpret_cast<uint2*>(const_cast<uint8_t*>(O.codes) + rr * kRowBytes + 8 * sub) = make_uint2(w0, w1);
        if (sub == 0) {
          *reinterpret_cast<uint32_t*>(const_cast<uint16_t*>(O.mins) + rr * (kD / kG)) = mp | (mp1 << 16);
          *reinterpret_cast<uint32_t*>(const_cast<uint16_t*>(O.scales) + rr * (kD / kG)) = sp | (sp1 << 16);
        }
      }
    }
  }
}

// ---------------------------------------------------------------- reconstruct (fast)
//
// Every warp finds the stored rows of its tile's tokens by itself: a dense
// loop stores token t at row t; a sparse loop stores the tile's present tokens
// in the compact rows tile_dir[k] .. tile_dir[k+1]-1, in token order, so the
// row of a present token is tile_dir[k] plus its rank in the tile's 64-bit
// presence mask (two warp OR-reductions over the tile's index slice). No
// block-wide barrier separates the items.

struct TileRows {
  unsigned long long mask;  // presence of tokens t0 .. t0 + 63 in the loop
  int c0;                   // stored row of the first present token
};

// Rows of tile k (tokens t0 = 64 k ..) in loop L, computed by a whole warp;
// an inconsistent directory entry yields an empty mask and sets bit 4.
__device__ __forceinline__ TileRows tile_rows(const CodecArgs& a, const LoopPlanes& L, int k, int nvalid, int lane) {
  TileRows r;
  if (!L.sparse) {
    r.mask = nvalid >= 64 ? ~0ull : ((1ull << nvalid) - 1ull);
    r.c0 = k * KVQ_TILE;
    return r;
  }
  const int c0 = __ldg(L.tile_dir + k), c1 = __ldg(L.tile_dir + k + 1);
  r.mask = 0;
  r.c0 = c0;
  if (c0 < 0 || c1 > L.n_rows || c0 > c1 || c1 - c0 > KVQ_TILE) {
    if (lane == 0 && a.err) atomicOr(a.err, 4);
    return r;
  }
  const int t0 = k * KVQ_TILE;
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i0 = 0; i0 < KVQ_TILE; i0 += 32) {
    const int c = c0 + i0 + lane;
    if (c < c1) {
      const int u = __ldg(L.active + c) - t0;
      if (u >= 0 && u < 32) lo |= 1u << u;
      else if (u >= 32 && u < KVQ_TILE) hi |= 1u << (u - 32);
      else if (a.err) atomicOr(a.err, 4);
    }
  }
  lo = __reduce_or_sync(0xffffffffu, lo);
  hi = __reduce_or_sync(0xffffffffu, hi);
  r.mask = (unsigned long long)hi << 32 | lo;
  return r;
}

// Stored row of token tt of the tile, or -1 if the loop holds no row for it.
__device__ __forceinline__ int row_in(const TileRows& r, int tt) {
  if (!((r.mask >> tt) & 1ull)) return -1;
  return r.c0 + __popcll(r.mask & ((1ull << tt) - 1ull));
}

// K parameters of the 16 channels 16 sub .. +15 of group `grp` of head h, loop L.
__device__ __forceinline__ void load_kpar16_global(const LoopPlanes& L, int h, int grp, int sub, float2* m, float2* s) {
  const long long pi = ((long long)h * L.kgroups + grp) * kD + 16 * sub;
  const uint4* mp = reinterpret_cast<const uint4*>(L.mins + pi);
  const uint4* sp = reinterpret_cast<const uint4*>(L.scales + pi);
  const uint4 m0 = __ldg(mp), m1 = __ldg(mp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
  const uint32_t mw[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
  const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    m[k] = fast::f16x2_to_f2(mw[k]);
    s[k] = fast::f16x2_to_f2(sw[k]);
  }
}

namespace fast {

// 16 channels of one stored row of an NVFP4 loop (codes cw, block scale sb, tensor
// scale st) as 8 BF16 pairs: RN_bf16(RN32(RN32(e2m1 * sb) * st)). The product
// e2m1 * sb carries at most 6 significant bits and lies in [2^-10, 2880] or is
// zero, so the FP16 pair product of the hardware-converted codes is that exact
// FP32 product.
__device__ __forceinline__ void dequant_nv16(uint2 cw, float sb, float st, uint32_t* out) {
  const __half2 sb2 = __float2half2_rn(sb);  // an E4M3 value: exact in FP16
  const uint32_t w[2] = {cw.x, cw.y};
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t e2 = e2m1x2_to_f16x2(w[h] >> (8 * k));
      const float2 p = __half22float2(__hmul2(*reinterpret_cast<const __half2*>(&e2), sb2));
      out[4 * h + k] = f2_to_bf2(make_float2(__fmul_rn(p.x, st), __fmul_rn(p.y, st)));
    }
}

// E2M1 codes of the pair (lo, hi) as one byte {lo in bits 0..3, hi in 4..7}, by
// the hardware conversion: nearest value, ties to the even code (the even
// mantissa), saturating at 6, the sign kept (zero included).
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u32.u8 %0, b;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

}  // namespace fast

// K: item = (64-token tile, head), 128 threads; eight lanes per token (lane
// `sub` = channels 16 sub .. +15) and four tokens per lane (16 w + 4 u + lg), so
// a lane loads each loop's parameters once for its four tokens (twice when a
// sparse loop's rows cross a group), and each token's output row (256 B) leaves
// in 16-byte stores.
constexpr int kReconKTok = 4;                             // tokens per lane
// (four 128-thread blocks per SM at 128 registers: faster than three at 159 despite a few spilled words)
constexpr int kReconKThreads = KVQ_TILE * 8 / kReconKTok;  // eight lanes per token, one tile per item

template <int DEPTH, bool kNv>
__global__ void __launch_bounds__(kReconKThreads, 4) reconstruct_k_fast_kernel(const __grid_constant__ CodecArgs a,
                                                                            const int32_t* prefix_ws) {
  using namespace fast;
  const int32_t* prefix = prefix_ws ? prefix_ws : a.one_prefix;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane & 7, lg = lane >> 3;
  const int H = a.H;
  __shared__ Chain C;

  const ItemRange ir = cta_items(prefix, a.n_requests);
  int cur_b = -1;
  for (long long it = ir.begin; it < ir.end; ++it) {
    const int b = owner_next(prefix, a.n_requests, it, cur_b);
    if (b != cur_b) {
      __syncthreads();  // every thread is done with the previous request's chain
      if (tid == 0) fill_chain(req_at(a, b), KVQ_K, DEPTH, H, C);
      __syncthreads();
      cur_b = b;
    }
    if (!kNv && C.any_nvfp4) {  // NVFP4 loops: the INT4-only instantiation refuses the request
      if (tid == 0 && a.err) atomicOr(a.err, 64);
      continue;
    }
    const int local = int(it - prefix[b]);
    const int k = local / H, h = local % H;
    const int t0 = k * KVQ_TILE;
    const int nvalid = min(KVQ_TILE, C.n_tokens - t0);
    uint16_t* out = a.reqs ? a.out[b] : a.one_out;
    if ((reinterpret_cast<uintptr_t>(out) & 15u) != 0) {
      if (tid == 0 && a.err) atomicOr(a.err, 16);
      continue;
    }
    int rows[kReconKTok][DEPTH];
    uint2 cw[kReconKTok][DEPTH];
#pragma unroll
    for (int j = 0; j < DEPTH; ++j) {
      const LoopPlanes& L = C.loop[j];
      const TileRows tr = tile_rows(a, L, k, nvalid, lane);
#pragma unroll
      for (int u = 0; u < kReconKTok; ++u) {
        const int tt = 4 * kReconKTok * warp + 4 * u + lg;
        rows[u][j] = tt < nvalid ? row_in(tr, tt) : -1;
        cw[u][j] = make_uint2(0, 0);
        if (rows[u][j] >= 0)
          cw[u][j] = __ldg(reinterpret_cast<const uint2*>(L.codes + ((long long)h * L.stride + rows[u][j]) * kRowBytes +
                                                          8 * sub));
      }
    }
    uint32_t acc[kReconKTok][8];
#pragma unroll
    for (int u = 0; u < kReconKTok; ++u)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[u][e] = 0;
#pragma unroll
    for (int j = 0; j < DEPTH; ++j) {
      const LoopPlanes& L = C.loop[j];
      if (kNv && L.fmt == KVQ_FMT_NVFP4) {  // NVFP4 residual: the lane's 16 channels are one block
        const float st = nvfp4_tensor_scale(L);
#pragma unroll
        for (int u = 0; u < kReconKTok; ++u) {
          const int row = rows[u][j];
          if (row < 0) continue;
          uint32_t dq[8];
          dequant_nv16(cw[u][j], nvfp4_block_scale(L, h, row, sub), st, dq);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[u][e] = bf2_add(acc[u][e], dq[e]);
        }
        continue;
      }
      float2 m[8], s[8];
      int cached = -1;
#pragma unroll
      for (int u = 0; u < kReconKTok; ++u) {
        const int row = rows[u][j];
        if (row < 0) continue;
        const int grp = L.ktile ? k : (row >> 6);  // tile grouping: the tile's own group
        if (grp != cached) {
          cached = grp;
          load_kpar16_global(L, h, cached, sub, m, s);
        }
        uint32_t dq[8];
        dequant_word_pp(cw[u][j].x, m, s, dq);
        dequant_word_pp(cw[u][j].y, m + 4, s + 4, dq + 4);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[u][e] = (j == 0) ? dq[e] : bf2_add(acc[u][e], dq[e]);
      }
    }
#pragma unroll
    for (int u = 0; u < kReconKTok; ++u) {
      const int tt = 4 * kReconKTok * warp + 4 * u + lg;
      if (tt < nvalid) {
        uint4* dst = reinterpret_cast<uint4*>(out + ((long long)(t0 + tt) * H + h) * kD + 16 * sub);
        dst[0] = make_uint4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
        dst[1] = make_uint4(acc[u][4], acc[u][5], acc[u][6], acc[u][7]);
      }
    }
  }
}

// V: item = 64-token tile (all heads); eight lanes per (token, head), lane
// `sub` = channels 16 sub .. +15; a warp takes four consecutive (token, head)
// pairs, i.e. 1 KB of contiguous output, and finds the tile's rows itself.
constexpr int kReconVFastThreads = 256;

template <int DEPTH, bool kNv>
__global__ void __launch_bounds__(kReconVFastThreads, 5) reconstruct_v_fast_kernel(const __grid_constant__ CodecArgs a,
                                                                                const int32_t* prefix_ws) {
  using namespace fast;
  constexpr int kWarps = kReconVFastThreads / 32;
  const int32_t* prefix = prefix_ws ? prefix_ws : a.one_prefix;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane & 7, lg = lane >> 3;
  const int H = a.H;
  __shared__ Chain C;

  const ItemRange ir = cta_items(prefix, a.n_requests);
  int cur_b = -1;
  for (long long it = ir.begin; it < ir.end; ++it) {
    const int b = owner_next(prefix, a.n_requests, it, cur_b);
    if (b != cur_b) {
      __syncthreads();  // every thread is done with the previous request's chain
      if (tid == 0) fill_chain(req_at(a, b), KVQ_V, DEPTH, H, C);
      __syncthreads();
      cur_b = b;
    }
    if (!kNv && C.any_nvfp4) {  // NVFP4 loops: the INT4-only instantiation refuses the request
      if (tid == 0 && a.err) atomicOr(a.err, 64);
      continue;
    }
    const int k = int(it - prefix[b]);
    const int t0 = k * KVQ_TILE;
    const int nvalid = min(KVQ_TILE, C.n_tokens - t0);
    uint16_t* out = a.reqs ? a.out[b] : a.one_out;
    if ((reinterpret_cast<uintptr_t>(out) & 15u) != 0) {
      if (tid == 0 && a.err) atomicOr(a.err, 16);
      continue;
    }
    TileRows tr[DEPTH];
#pragma unroll
    for (int j = 0; j < DEPTH; ++j) tr[j] = tile_rows(a, C.loop[j], k, nvalid, lane);
    const int npairs = nvalid * H;
    for (int q4 = warp; q4 * 4 < npairs; q4 += kWarps) {
      const int pr = q4 * 4 + lg;
      const bool live = pr < npairs;
      const int tt = live ? pr / H : 0, h = live ? pr % H : 0;
      uint2 cw[DEPTH];
      uint32_t m16[DEPTH], s16[DEPTH];
      bool have[DEPTH];
#pragma unroll
      for (int j = 0; j < DEPTH; ++j) {
        const int row = live ? row_in(tr[j], tt) : -1;
        have[j] = row >= 0;
        cw[j] = make_uint2(0, 0);
        m16[j] = s16[j] = 0;
        if (have[j]) {
          const LoopPlanes& L = C.loop[j];
          const long long rr = (long long)h * L.stride + row;
          cw[j] = __ldg(reinterpret_cast<const uint2*>(L.codes + rr * kRowBytes + 8 * sub));
          if (kNv && L.fmt == KVQ_FMT_NVFP4) {  // E4M3 block scale of the lane's block; the tensor scale
            m16[j] = __ldg(reinterpret_cast<const uint8_t*>(L.mins) + rr * (kD / 16) + sub);
            s16[j] = __float_as_uint(nvfp4_tensor_scale(L));
          } else {
            m16[j] = __ldg(L.mins + rr * (kD / kG) + (sub >> 2));
            s16[j] = __ldg(L.scales + rr * (kD / kG) + (sub >> 2));
          }
        }
      }
      uint32_t acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0;
#pragma unroll
      for (int j = 0; j < DEPTH; ++j) {
        if (!have[j]) continue;
        uint32_t dq[8];
        if (kNv && C.loop[j].fmt == KVQ_FMT_NVFP4) {
          dequant_nv16(cw[j], e4m3_to_f32(m16[j]), __uint_as_float(s16[j]), dq);
        } else {
          const float mf = f16_bits_to_f32(uint16_t(m16[j])), sf = f16_bits_to_f32(uint16_t(s16[j]));
          dequant_word(cw[j].x, make_float2(mf, mf), make_float2(sf, sf), dq);
          dequant_word(cw[j].y, make_float2(mf, mf), make_float2(sf, sf), dq + 4);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = (j == 0) ? dq[e] : bf2_add(acc[e], dq[e]);
      }
      if (live) {
        uint4* dst = reinterpret_cast<uint4*>(out + ((long long)(t0 + tt) * H + h) * kD + 16 * sub);
        dst[0] = make_uint4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_uint4(acc[4], acc[5], acc[6], acc[7]);
      }
    }
  }
}

// ---------------------------------------------------------------- NVFP4 residual encode (fast, chains up to 4 loops)
//
// The two NVFP4 passes of a residual loop r <= 3 in the layout of the fast V
// encoder: item = 64 stored rows (all heads), eight lanes per (row, head), lane
// `sub` = channels 16 sub .. 16 sub + 15 = exactly one NVFP4 block, so a block's
// max |delta| is lane-local. The predecessor chain is decoded per loop in its own
// format (INT4 K, INT4 V, or NVFP4). Codes come from the hardware E2M1
// conversion of the product delta * RN32(1 / e_b); a pair whose product lies
// within 2^-20 (relative) of an E2M1 decision boundary takes the IEEE quotients,
// the definition's, instead.


// Five resident blocks per SM (a few spilled words): 17% faster than three, 3% faster than four.
template <int R, bool kAmax>
__global__ void __launch_bounds__(kEncVFastThreads, 5) nvfp4_encode_fast_kernel(const __grid_constant__ CodecArgs a,
                                                                             const int32_t* prefix_ws) {
  using namespace fast;
  constexpr int RA = R > 0 ? R : 1;
  constexpr int kWarps = kEncVFastThreads / 32;
  const int32_t* prefix = prefix_ws ? prefix_ws : a.one_prefix;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane & 7, lg = lane >> 3;
  const int H = a.H;
  __shared__ Chain C;
  __shared__ int s_tok[kG];
  __shared__ int s_row[RA][kG];

  const ItemRange ir = cta_items(prefix, a.n_requests);
  int cur_b = -1;
  for (long long it = ir.begin; it < ir.end; ++it) {
    const int b = owner_next(prefix, a.n_requests, it, cur_b);
    if (b != cur_b) {
      __syncthreads();  // every thread is done with the previous request's chain
      if (threadIdx.x == 0) fill_chain(req_at(a, b), a.kind, R + 1, H, C);
      cur_b = b;
    }
    __syncthreads();
    const LoopPlanes& O = C.loop[R];
    if (R < 1 || O.fmt != KVQ_FMT_NVFP4) {  // the table does not hold an NVFP4 residual here
      if (threadIdx.x == 0 && a.err) atomicOr(a.err, 64);
      continue;
    }
    const int n = O.n_rows;
    const int r0 = int(it - prefix[b]) * kG;
    const int len = min(kG, n - r0);
    const uint16_t* x = source_of(a, b);
    if (threadIdx.x < len) {
      const int t = O.sparse ? __ldg(O.active + r0 + threadIdx.x) : r0 + threadIdx.x;
      s_tok[threadIdx.x] = t;
#pragma unroll
      for (int j = 0; j < R; ++j) s_row[j][threadIdx.x] = row_of(C.loop[j], t);
    }
    __syncthreads();
    if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0) {
      if (threadIdx.x == 0 && a.err) atomicOr(a.err, 16);
      continue;
    }
    float* rec = reinterpret_cast<float*>(const_cast<uint16_t*>(O.scales));
    float st = 0.0f, six_st = 0.0f;
    bool all_zero = true;
    if (!kAmax) {
      const float amax = rec[1];
      all_zero = !(amax > 0.0f);
      st = __fdiv_rn(amax, 2688.0f);
      six_st = __fmul_rn(6.0f, st);
    }
    float wmax = 0.0f;
    const int nquads = H * (kG / 4);
    for (int qd = warp; qd < nquads; qd += kWarps) {
      const int h = qd / (kG / 4);
      const int i = (qd % (kG / 4)) * 4 + lg;
      const bool live = i < len;
      uint32_t d[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (live) {
        const int t = s_tok[i];
        const uint4* src = reinterpret_cast<const uint4*>(x + ((long long)t * H + h) * kD + 16 * sub);
        const uint4 xa = __ldg(src), xb = __ldg(src + 1);
        const uint32_t xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        uint32_t acc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = 0u;
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const int row = s_row[j][i];
          if (row < 0) continue;  // absent: the predecessor inherits
          const LoopPlanes& L = C.loop[j];
          const long long rr = (long long)h * L.stride + row;
          const uint2 cw = __ldg(reinterpret_cast<const uint2*>(L.codes + rr * kRowBytes + 8 * sub));
          uint32_t dq[8];
          if (L.fmt == KVQ_FMT_NVFP4) {
            dequant_nv16(cw, nvfp4_block_scale(L, h, row, sub), nvfp4_tensor_scale(L), dq);
          } else if (a.kind == KVQ_K) {
            float2 m[8], s[8];
            load_kpar16_global(L, h, k_group(L, t, row), sub, m, s);
            dequant_word_pp(cw.x, m, s, dq);
            dequant_word_pp(cw.y, m + 4, s + 4, dq + 4);
          } else {
            const float mf = f16_bits_to_f32(__ldg(L.mins + rr * (kD / kG) + (sub >> 2)));
            const float sf = f16_bits_to_f32(__ldg(L.scales + rr * (kD / kG) + (sub >> 2)));
            dequant_word(cw.x, make_float2(mf, mf), make_float2(sf, sf), dq);
            dequant_word(cw.y, make_float2(mf, mf), make_float2(sf, sf), dq + 4);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[k] = (j == 0) ? dq[k] : bf2_add(acc[k], dq[k]);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) d[k] = bf2_sub(xv[k], acc[k]);
      }
      // the block's max |delta| (BF16 pairs with the sign bits cleared)
      uint32_t am2 = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k) am2 = bf2_max(am2, d[k] & 0x7FFF7FFFu);
      const float ab = fmaxf(bf_lo(am2), bf_hi(am2));
      if (kAmax) {
        wmax = fmaxf(wmax, ab);
        continue;
      }
      const uint32_t sb = all_zero ? 0u : f32_to_e4m3(__fdiv_rn(ab, six_st));
      const float eb = __fmul_rn(e4m3_to_f32(sb), st);
      // the product y = delta * RN32(1 / e_b) lies within 2^-22 (relative) of the
      // quotient while 1 / e_b is a normal number; a pair whose codes change when y
      // moves by 2^-20 (relative) lies near a decision boundary and takes the IEEE
      // quotients instead
      const float rc = eb != 0.0f ? __frcp_rn(eb) : 0.0f;
      const bool by_div = !(fabsf(rc) >= 1.17549435e-38f && fabsf(rc) <= 3.0e38f);
      constexpr float kUp = 1.00000095367431640625f, kDn = 0.99999904632568359375f;  // 1 +- 2^-20
      uint32_t w[2] = {0u, 0u};
      if (eb != 0.0f) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float v0 = bf_lo(d[k]), v1 = bf_hi(d[k]);
          const float y0 = __fmul_rn(v0, rc), y1 = __fmul_rn(v1, rc);
          uint32_t c = f32x2_to_e2m1x2(y0, y1);
          const uint32_t cu = f32x2_to_e2m1x2(__fmul_rn(y0, kUp), __fmul_rn(y1, kUp));
          const uint32_t cd = f32x2_to_e2m1x2(__fmul_rn(y0, kDn), __fmul_rn(y1, kDn));
          if (by_div || c != cu || c != cd) c = f32x2_to_e2m1x2(__fdiv_rn(v0, eb), __fdiv_rn(v1, eb));
          w[k >> 2] |= c << (8 * (k & 3));
        }
      }
      if (live) {
        const long long rr = (long long)h * O.stride + r0 + i;
        *reinterpret_cast<uint2*>(const_cast<uint8_t*>(O.codes) + rr * kRowBytes + 8 * sub) = make_uint2(w[0], w[1]);
        reinterpret_cast<uint8_t*>(const_cast<uint16_t*>(O.mins))[rr * (kD / 16) + sub] = uint8_t(sb);
      }
    }
    if (kAmax) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
      if (lane == 0 && wmax > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(rec + 1), __float_as_uint(wmax));
      wmax = 0.0f;
    } else if (r0 == 0 && threadIdx.x == 0) {
      rec[0] = st;  // the stream's tensor scale, once
    }
  }
}

// ---------------------------------------------------------------- tile append: index planes

// One block per loop. A position outside [0, 64), or not ascending, sets bit 4
// and is replaced by a valid ascending list, so the encode that follows stays
// inside the tile.
__global__ void __launch_bounds__(64) append_index_kernel(const __grid_constant__ AppendIndexArgs a) {
  const AppendIndexArgs::Loop& L = a.loop[blockIdx.x];
  if (L.rel == nullptr) return;  // dense loop: no index
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const int i = threadIdx.x;
  int v = 0;
  if (i < L.n_new) {
    v = __ldg(L.rel + i);
    const int prev = i > 0 ? __ldg(L.rel + i - 1) : -1;
    if (v < 0 || v >= KVQ_TILE || v <= prev) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    v = i;  // 0 .. n_new - 1
    if (i == 0 && a.err) atomicOr(a.err, 4);
  }
  if (i < L.n_new) {
    L.rel_ws[i] = v;
    L.active[L.n_old + i] = a.T + v;
  }
  if (i == 0) {
    L.dir_ws[0] = 0;
    L.dir_ws[1] = L.n_new;
    L.tile_dir[a.T / KVQ_TILE] = L.n_old;
    L.tile_dir[a.T / KVQ_TILE + 1] = L.n_old + L.n_new;
  }
}

cudaError_t launch_append_index(const AppendIndexArgs& a, cudaStream_t stream) {
  append_index_kernel<<<a.n_loops, 64, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

// ---------------------------------------------------------------- batched tile append: checks, index, table

// One thread per request: the request can take the tile (whole tiles so far,
// every loop INT4 with room for the tile, a dense base, sparse loops under
// tile grouping with 0..64 positions, dense loops with all 64).
__global__ void __launch_bounds__(256) append_check_kernel(const __grid_constant__ AppendBatchArgs a) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.n_requests) return;
  const kvq_request& R = a.reqs[b];
  bool ok = R.n_tokens >= 0 && R.n_tokens % KVQ_TILE == 0 && R.n_loops == a.n_loops;
  for (int j = 0; ok && j < a.n_loops; ++j) {
    const kvq_loop_ref& L = R.loop[j];
    const int m = a.n_tile_active[j * a.n_requests + b];
    const int32_t* rel = a.tile_active[j * a.n_requests + b];
    ok = !(L.flags & (KVQ_LOOP_K_NVFP4 | KVQ_LOOP_V_NVFP4)) && L.row_cap > 0 && L.n_rows + m <= L.row_cap &&
         R.n_tokens / KVQ_TILE < L.kgroup_cap && L.k_codes && L.k_mins && L.k_scales && L.v_codes && L.v_mins &&
         L.v_scales;
    if (L.active_idx == nullptr)
      ok = ok && rel == nullptr && m == KVQ_TILE && L.n_rows == R.n_tokens;
    else
      ok = ok && j > 0 && rel != nullptr && m >= 0 && m <= KVQ_TILE && (L.flags & KVQ_LOOP_K_TILE) && L.tile_dir;
  }
  a.skip[b] = ok ? 0 : 1;
  if (!ok) atomicOr(a.err, 1);
}

// Block (request, loop), 64 threads: a sparse loop's positions (checked: a bad
// list sets bit 4 and is replaced by 0 .. m-1) become absolute indices after the
// stored rows, the tile directory gains the tile, and K groups of tiles without
// stored rows get +0 parameters.
__global__ void __launch_bounds__(64) append_index_batch_kernel(const __grid_constant__ AppendBatchArgs a) {
  const int b = blockIdx.x, j = blockIdx.y;
  if (a.skip[b]) return;
  const kvq_request& R = a.reqs[b];
  const kvq_loop_ref& L = R.loop[j];
  if (L.active_idx == nullptr) return;
  const int T = R.n_tokens, k = T / KVQ_TILE, n_old = L.n_rows;
  const int m = a.n_tile_active[j * a.n_requests + b];
  const int32_t* rel = a.tile_active[j * a.n_requests + b];
  __shared__ int s_bad;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const int i = threadIdx.x;
  int v = 0;
  if (i < m) {
    v = rel[i];
    const int prev = i > 0 ? rel[i - 1] : -1;
    if (v < 0 || v >= KVQ_TILE || v <= prev) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    v = i;
    if (i == 0) atomicOr(a.err, 4);
  }
  if (i < m) const_cast<int32_t*>(L.active_idx)[n_old + i] = T + v;
  if (i == 0) {
    L.tile_dir[k] = n_old;
    L.tile_dir[k + 1] = n_old + m;
  }
  int g0 = 0, g1 = 0;  // K groups to clear (tile grouping: a tile without stored rows)
  if (m == 0 && n_old > 0) g0 = k, g1 = k + 1;
  if (m > 0 && n_old == 0) g0 = 0, g1 = k;
  const int per = (g1 - g0) * kD;
  for (int x = i; x < a.H * per; x += blockDim.x) {
    const int h = x / per, r = x % per;
    const long long pi = ((long long)h * L.kgroup_cap + g0) * kD + r;
    L.k_mins[pi] = 0;
    L.k_scales[pi] = 0;
  }
}

// One thread per request: the table counts the tile.
__global__ void __launch_bounds__(256) append_table_kernel(const __grid_constant__ AppendBatchArgs a) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.n_requests || a.skip[b]) return;
  kvq_request& R = a.reqs[b];
  for (int j = 0; j < a.n_loops; ++j) R.loop[j].n_rows += a.n_tile_active[j * a.n_requests + b];
  R.n_tokens += KVQ_TILE;
}

cudaError_t launch_append_batch_prep(const AppendBatchArgs& a, cudaStream_t stream) {
  const int blocks = (a.n_requests + 255) / 256;
  append_check_kernel<<<blocks, 256, 0, stream>>>(a);
  count_launch();
  append_index_batch_kernel<<<dim3(a.n_requests, a.n_loops), 64, 0, stream>>>(a);
  count_launch();
  append_table_kernel<<<blocks, 256, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

// ---------------------------------------------------------------- launchers

static int single_items(const CodecArgs& a, int mode) {
  const kvq_request& R = a.one;
  const int n = R.loop[a.loop < KVQ_MAX_LOOPS ? a.loop : 0].n_rows;
  switch (mode) {
    case kModeNvAmax:
    case kModeNvEnc: return (n + kG - 1) / kG;
    case kModeEncK: {
      const kvq_loop_ref& L = R.loop[a.loop < KVQ_MAX_LOOPS ? a.loop : 0];
      return a.H * k_groups_of((L.flags & KVQ_LOOP_K_TILE) != 0, n, R.n_tokens);
    }
    case kModeEncV: return (n + kG - 1) / kG;
    case kModeTileDir: return R.loop[a.loop].active_idx ? (R.n_tokens + KVQ_TILE - 1) / KVQ_TILE + 1 : 0;
    case kModeReconK: return ((R.n_tokens + KVQ_TILE - 1) / KVQ_TILE) * a.H;
    default: return (R.n_tokens + KVQ_TILE - 1) / KVQ_TILE;
  }
}

cudaError_t launch_codec(const CodecArgs& a_in, int mode, int32_t* prefix_ws, int sms, cudaStream_t stream) {
  CodecArgs a = a_in;
  // NVFP4 loops (bit j of a.nvfp4: loop j): an NVFP4 output loop takes the two
  // NVFP4 passes; an INT4 output loop or a reconstruction whose chain holds an
  // NVFP4 loop takes the any-depth kernels, which decode either format.
  const uint32_t below = a.loop >= 32 ? 0xFFFFFFFFu : ((1u << a.loop) - 1u);  // loops 0 .. loop-1
  const bool nv_out = (mode == kModeEncK || mode == kModeEncV) && a.loop < 32 && ((a.nvfp4 >> a.loop) & 1u);
  const bool nv_chain = (a.nvfp4 & below) != 0;
  if (nv_out) mode = kModeNvAmax;
  // K reconstruction of INT4 chains up to 4 loops runs one item per (tile, head)
  if (mode == kModeRecon && a.kind == KVQ_K && a.loop >= 1 && a.loop <= kFastMaxDepth) mode = kModeReconK;
  const int32_t* prefix = nullptr;  // nullptr: kernels read a.one_prefix
  long long items = -1;             // -1: known only on the device
  if (a.reqs == nullptr) {
    a.n_requests = 1;
    a.one_prefix[0] = 0;
    a.one_prefix[1] = single_items(a, mode);
    items = a.one_prefix[1];
    if (items == 0) return cudaSuccess;
  } else {
    if (a.n_requests == 0) return cudaSuccess;
    items_plan_kernel<<<1, 1024, 0, stream>>>(a, mode, prefix_ws);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prefix = prefix_ws;
  }
  // a fixed grid of as many CTAs as fit on the GPU, fewer when a single
  // request has fewer items
  auto grid_for = [&](int per_sm) {
    long long cap = (long long)per_sm * sms;
    return int(items >= 0 && items < cap ? items : cap);
  };
  // Fast kernels: four waves of resident blocks, so that blocks finishing early
  // take the remaining items and kernels on other streams can interleave.
  auto run = [&](auto kern, int threads) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    kern<<<grid_for(4 * per_sm), threads, 0, stream>>>(a, prefix);
  };
  switch (mode) {
    case kModeNvAmax:
      switch (a.loop) {  // residual loops of chains up to 4 loops: the fast passes
        case 1:
          run(nvfp4_encode_fast_kernel<1, true>, kEncVFastThreads);
          count_launch();
          run(nvfp4_encode_fast_kernel<1, false>, kEncVFastThreads);
          break;
        case 2:
          run(nvfp4_encode_fast_kernel<2, true>, kEncVFastThreads);
          count_launch();
          run(nvfp4_encode_fast_kernel<2, false>, kEncVFastThreads);
          break;
        case 3:
          run(nvfp4_encode_fast_kernel<3, true>, kEncVFastThreads);
          count_launch();
          run(nvfp4_encode_fast_kernel<3, false>, kEncVFastThreads);
          break;
        default:
          nvfp4_encode_kernel<true><<<grid_for(4), kEncVThreads, 0, stream>>>(a, prefix);
          count_launch();
          nvfp4_encode_kernel<false><<<grid_for(4), kEncVThreads, 0, stream>>>(a, prefix);
          break;
      }
      break;
    case kModeEncK:
      switch (nv_chain ? -1 : a.loop) {
        case 0: run(encode_k_fast_kernel<0>, kEncKThreads); break;
        case 1: run(encode_k_fast_kernel<1>, kEncKThreads); break;
        case 2: run(encode_k_fast_kernel<2>, kEncKThreads); break;
        case 3: run(encode_k_fast_kernel<3>, kEncKThreads); break;
        default: encode_k_generic_kernel<<<grid_for(8), kD, 0, stream>>>(a, prefix); break;
      }
      break;
    case kModeEncV:
      switch (nv_chain ? -1 : a.loop) {
        case 0: run(encode_v_fast_kernel<0>, kEncVFastThreads); break;
        case 1: run(encode_v_fast_kernel<1>, kEncVFastThreads); break;
        case 2: run(encode_v_fast_kernel<2>, kEncVFastThreads); break;
        case 3: run(encode_v_fast_kernel<3>, kEncVFastThreads); break;
        default: encode_v_generic_kernel<<<grid_for(4), kEncVThreads, 0, stream>>>(a, prefix); break;
      }
      break;
    case kModeTileDir: {
      long long blocks = items >= 0 ? (items + 255) / 256 : 2LL * sms;
      if (blocks > 2LL * sms) blocks = 2LL * sms;
      tile_dir_kernel<<<int(blocks), 256, 0, stream>>>(a, prefix);
      break;
    }
    case kModeReconK:  // (a loop-1 chain is the INT4 base alone)
      switch (a.loop + (nv_chain && a.loop >= 2 ? 8 : 0)) {
        case 1: run(reconstruct_k_fast_kernel<1, false>, kReconKThreads); break;
        case 2: run(reconstruct_k_fast_kernel<2, false>, kReconKThreads); break;
        case 3: run(reconstruct_k_fast_kernel<3, false>, kReconKThreads); break;
        case 4: run(reconstruct_k_fast_kernel<4, false>, kReconKThreads); break;
        case 8 + 2: run(reconstruct_k_fast_kernel<2, true>, kReconKThreads); break;
        case 8 + 3: run(reconstruct_k_fast_kernel<3, true>, kReconKThreads); break;
        default: run(reconstruct_k_fast_kernel<4, true>, kReconKThreads); break;
      }
      break;
    default:
      if (a.kind == KVQ_V && a.loop >= 1 && a.loop <= kFastMaxDepth) {
        switch (a.loop + (nv_chain && a.loop >= 2 ? 8 : 0)) {
          case 1: run(reconstruct_v_fast_kernel<1, false>, kReconVFastThreads); break;
          case 2: run(reconstruct_v_fast_kernel<2, false>, kReconVFastThreads); break;
          case 3: run(reconstruct_v_fast_kernel<3, false>, kReconVFastThreads); break;
          case 4: run(reconstruct_v_fast_kernel<4, false>, kReconVFastThreads); break;
          case 8 + 2: run(reconstruct_v_fast_kernel<2, true>, kReconVFastThreads); break;
          case 8 + 3: run(reconstruct_v_fast_kernel<3, true>, kReconVFastThreads); break;
          default: run(reconstruct_v_fast_kernel<4, true>, kReconVFastThreads); break;
        }
      } else {
        reconstruct_generic_kernel<<<grid_for(4), kReconThreads, 0, stream>>>(a, prefix);
      }
      break;
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvq
