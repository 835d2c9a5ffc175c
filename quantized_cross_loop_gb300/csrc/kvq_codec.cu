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

__device__ __forceinline__ int items_of(const CodecArgs& a, const kvq_request& R, int mode) {
  if (R.n_tokens < 0 || R.n_loops > KVQ_MAX_LOOPS) return 0;
  switch (mode) {
    case kModeEncK: {
      if (a.loop >= R.n_loops) return 0;
      int n = R.loop[a.loop].n_rows;
      return n > 0 ? a.H * ((n + kG - 1) / kG) : 0;
    }
    case kModeEncV: {
      if (a.loop >= R.n_loops) return 0;
      int n = R.loop[a.loop].n_rows;
      return (n + kG - 1) / kG;
    }
    case kModeTileDir: {
      if (a.loop >= R.n_loops || R.loop[a.loop].active_idx == nullptr) return 0;
      return (R.n_tokens + KVQ_TILE - 1) / KVQ_TILE + 1;
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
    int v = b < a.n_requests ? items_of(a, req_at(a, b), mode) : 0;
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

// One thread fills the chain of loops 0..n-1 of request R for `kind`.
__device__ void fill_chain(const kvq_request& R, int kind, int n, int H, Chain& C) {
  C.depth = n;
  C.kind = kind;
  C.n_tokens = R.n_tokens;
  C.n_heads = H;
  for (int j = 0; j < n; ++j) {
    const kvq_loop_ref& L = R.loop[j];
    LoopPlanes& P = C.loop[j];
    P.n_rows = L.n_rows;
    P.sparse = L.active_idx != nullptr;
    P.active = L.active_idx;
    P.tile_dir = L.tile_dir;
    P.codes = kind == KVQ_K ? L.k_codes : L.v_codes;
    P.mins = kind == KVQ_K ? L.k_mins : L.v_mins;
    P.scales = kind == KVQ_K ? L.k_scales : L.v_scales;
  }
}

__device__ __forceinline__ const uint16_t* source_of(const CodecArgs& a, int b) {
  return a.reqs ? a.x[b] : a.one_x;
}

// ---------------------------------------------------------------- encode K

__global__ void __launch_bounds__(kD) encode_k_kernel(const __grid_constant__ CodecArgs a, const int32_t* prefix_ws) {
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
    const int local = int(it - prefix[b]);
    const int g = local / H, h = local % H;
    const LoopPlanes& O = C.loop[r];
    const int n = O.n_rows;
    const int r0 = g * kG;
    const int len = min(kG, n - r0);
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
          val = round_bf16(__fsub_rn(xv, chain1(C, r, rows, h, d)));
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
    long long pi = ((long long)h * ((n + kG - 1) / kG) + g) * kD + d;
    const_cast<uint16_t*>(O.mins)[pi] = f32_to_f16_bits(mn);
    const_cast<uint16_t*>(O.scales)[pi] = f32_to_f16_bits(s32);
    __syncthreads();
    // len rows x 64 bytes, contiguous in the head-major plane: 16-byte stores.
    uint4* dst = reinterpret_cast<uint4*>(const_cast<uint8_t*>(O.codes) + ((long long)h * n + r0) * kRowBytes);
    const uint4* src = reinterpret_cast<const uint4*>(&s_codes[0][0]);
    for (int k = d; k < len * (kRowBytes / 16); k += blockDim.x) dst[k] = src[k];
  }
}

// ---------------------------------------------------------------- encode V

constexpr int kEncVThreads = 256;

__global__ void __launch_bounds__(kEncVThreads) encode_v_kernel(const __grid_constant__ CodecArgs a,
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
        chain4(C, r, rows, h, c0, xh);
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
      *reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(O.codes) + ((long long)h * n + row) * kRowBytes + lane * 2) =
          packed;
      if ((lane & 15) == 0) {
        long long pi = ((long long)h * n + row) * (kD / kG) + (lane >> 4);
        const_cast<uint16_t*>(O.mins)[pi] = f32_to_f16_bits(mn);
        const_cast<uint16_t*>(O.scales)[pi] = f32_to_f16_bits(s32);
      }
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

__global__ void __launch_bounds__(kReconThreads) reconstruct_kernel(const __grid_constant__ CodecArgs a,
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
      chain4(C, depth, rows, h, lane * 4, v);
      uint2 o;
      o.x = uint32_t(f32_to_bf16_bits(v[0])) | (uint32_t(f32_to_bf16_bits(v[1])) << 16);
      o.y = uint32_t(f32_to_bf16_bits(v[2])) | (uint32_t(f32_to_bf16_bits(v[3])) << 16);
      *reinterpret_cast<uint2*>(out + ((long long)(t0 + tt) * H + h) * kD + lane * 4) = o;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- launchers

static int single_items(const CodecArgs& a, int mode) {
  const kvq_request& R = a.one;
  const int n = R.loop[a.loop < KVQ_MAX_LOOPS ? a.loop : 0].n_rows;
  switch (mode) {
    case kModeEncK: return n > 0 ? a.H * ((n + kG - 1) / kG) : 0;
    case kModeEncV: return (n + kG - 1) / kG;
    case kModeTileDir: return R.loop[a.loop].active_idx ? (R.n_tokens + KVQ_TILE - 1) / KVQ_TILE + 1 : 0;
    default: return (R.n_tokens + KVQ_TILE - 1) / KVQ_TILE;
  }
}

cudaError_t launch_codec(const CodecArgs& a_in, int mode, int32_t* prefix_ws, int sms, cudaStream_t stream) {
  CodecArgs a = a_in;
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
  // a fixed grid of a few CTAs per SM, fewer when a single request has fewer items
  auto grid_for = [&](int per_sm) {
    long long cap = (long long)per_sm * sms;
    return int(items >= 0 && items < cap ? items : cap);
  };
  switch (mode) {
    case kModeEncK: encode_k_kernel<<<grid_for(8), kD, 0, stream>>>(a, prefix); break;
    case kModeEncV: encode_v_kernel<<<grid_for(4), kEncVThreads, 0, stream>>>(a, prefix); break;
    case kModeTileDir: {
      long long blocks = items >= 0 ? (items + 255) / 256 : 2LL * sms;
      if (blocks > 2LL * sms) blocks = 2LL * sms;
      tile_dir_kernel<<<int(blocks), 256, 0, stream>>>(a, prefix);
      break;
    }
    default: reconstruct_kernel<<<grid_for(4), kReconThreads, 0, stream>>>(a, prefix); break;
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvq
