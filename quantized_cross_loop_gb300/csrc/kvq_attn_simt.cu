// kvq_attn_simt.cu — plan and combine kernels, and the CUDA-core decode
// attention kernel over packed K/V.
//
// FlashLoop RFC (vllm-rlt issue #156) §3.2: historical K/V are read at the
// requested depth and reconstructed if compressed; scores use 1/sqrt(head_dim);
// §5: FP32 mass and accumulation; §3.3: readers consume the packed base and
// residual tiles directly (no BF16 shadow cache in HBM).
//
// The CUDA-core kernel decodes each 64-token tile of K and V into shared memory
// with the FP32 chain (dequantised values summed in FP32, the values a direct
// packed reader works with), then runs FP32 dot products, an online softmax
// and the PV sum. It is the design the tensor-core kernel is measured against.
#include "kvq_attn_common.cuh"

namespace kvq {

// ---------------------------------------------------------------- plan

__global__ void __launch_bounds__(1024) plan_kernel(AttnArgs a) {
  __shared__ long long s_carry;
  __shared__ int s_warp[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  allow_dependents();  // the attention kernel may start its prologue; it waits for this grid before reading the plan
  if (threadIdx.x == 0) {
    s_carry = 0;
    a.prefix[0] = 0;
    if (a.clear_err) {
      *a.err = 0;
      *a.flags = 0;
    }
  }
  __syncthreads();
  for (int base = 0; base < a.n_requests; base += blockDim.x) {
    int b = base + threadIdx.x;
    int v = 0;
    if (b < a.n_requests) {
      const kvq_request& r = a.reqs[b];
      if (!request_ok(r, a.depth)) {
        atomicOr(a.err, 1);
      } else if (nvfp4_refused(a, r)) {
        atomicOr(a.err, 64);
      } else {
        v = a.H * n_tiles_of(r.n_tokens);
        if (r.n_sink + r.n_tail > 0) atomicOr(a.flags, 1);
        if (holds_nvfp4(r, a.depth)) atomicOr(a.flags, 2);
      }
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
    if (incl > 0x7FFFFFFFLL) {  // more than 2^31 - 1 tiles in one call
      atomicOr(a.err, 2);
      incl = 0x7FFFFFFFLL;
    }
    if (b < a.n_requests) a.prefix[b + 1] = int(incl);
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_carry = incl;
    __syncthreads();
  }
}

cudaError_t launch_plan(const AttnArgs& a, cudaStream_t stream) {
  plan_kernel<<<1, 1024, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

// ---------------------------------------------------------------- combine

// Grid-stride over (request, KV head, query head) items. Most need nothing:
// their unit's tile range lies inside one CTA's, which wrote the output
// directly; that is decided from the tile prefix alone. A request with no
// tiles is read only to tell a refused entry (NaN output) from one without
// packed tokens (zero output and an empty softmax state). A split unit's
// query heads are merged by separate blocks, each slot loop unrolled so that
// the slots' loads overlap.
__global__ void __launch_bounds__(kD) combine_kernel(AttnArgs a) {
  wait_prior_grid();
  allow_dependents();
  const int d = threadIdx.x;
  const int g = a.g;
  const long long W = a.prefix[a.n_requests];
  const int C = a.n_ctas;
  const long long items = (long long)a.n_requests * a.H * g;
  for (long long it = blockIdx.x; it < items; it += gridDim.x) {
    const int u = int(it / g), i = int(it % g);
    const int b = u / a.H, h = u % a.H;
    float* outp = a.out + ((long long)b * a.Hq + (long long)h * g + i) * kD;
    float2* stats = a.stats + (long long)b * a.Hq + (long long)h * g + i;
    const int p0 = a.prefix[b], p1 = a.prefix[b + 1];
    if (p1 <= p0) {
      const bool ok = attn_request_ok(a, a.reqs[b]);
      outp[d] = ok ? 0.0f : __int_as_float(0x7fc00000);
      if (ok && d == 0) *stats = make_float2(-INFINITY, 0.0f);  // no packed tokens: an empty softmax state
      continue;
    }
    const int nt = (p1 - p0) / a.H;
    const long long s = (long long)p0 + (long long)h * nt;
    const long long e = s + nt;
    const int c_lo = cta_of(s, W, C), c_hi = cta_of(e - 1, W, C);
    if (c_lo == c_hi) continue;  // written directly by its only CTA
    float M = -INFINITY;
#pragma unroll 4
    for (int c = c_lo; c <= c_hi; ++c) {
      if (cta_start(c, W, C) == cta_start(c + 1, W, C)) continue;  // empty range
      M = fmaxf(M, a.partials[(size_t)(c + u) * kSlotFloats + i]);
    }
    float L = 0.0f, acc = 0.0f;
#pragma unroll 4
    for (int c = c_lo; c <= c_hi; ++c) {
      if (cta_start(c, W, C) == cta_start(c + 1, W, C)) continue;
      const float* slot = a.partials + (size_t)(c + u) * kSlotFloats;
      const float m = slot[i];
      const float w = (m == -INFINITY) ? 0.0f : exp2f(m - M);
      L += slot[kMaxG + i] * w;
      acc += slot[2 * kMaxG + i * kD + d] * w;
    }
    outp[d] = acc / L;
    if (d == 0) *stats = make_float2(M, L);
  }
}

// Blocks of the grid-stride kernels below: the unit count, capped at two
// blocks per attention CTA.
static int unit_grid(const AttnArgs& a) {
  const long long units = (long long)a.n_requests * a.H;
  const long long cap = 2LL * (a.n_ctas > 0 ? a.n_ctas : 1);
  return int(units < cap ? units : cap);
}

cudaError_t launch_combine(const AttnArgs& a, cudaStream_t stream) {
  if (a.n_requests == 0) return cudaSuccess;
  const long long items = (long long)a.n_requests * a.H * a.g;
  const long long cap = 4LL * (a.n_ctas > 0 ? a.n_ctas : 1);
  cudaError_t e = launch_dependent(combine_kernel, dim3(unsigned(items < cap ? items : cap)), dim3(kD), 0, stream, a);
  count_launch();
  return e;
}

// ---------------------------------------------------------------- BF16 segments
//
// One block per (request, KV head): the request's BF16 sink and tail tokens are
// attended in FP32 (log2 domain) — each warp takes every fourth token, a lane
// four channels, and keeps its own online softmax over its tokens; the four
// are merged, then combined by log-sum-exp with the packed part's result and
// its (max, sum) state.

constexpr int kSegWarps = 4;
constexpr float kSegLog2e = 1.4426950408889634f;

// Grid-stride over the (request, KV head) units; the whole grid leaves at once
// when the plan saw no request with segments.
__global__ void __launch_bounds__(32 * kSegWarps) segment_kernel(AttnArgs a) {
  wait_prior_grid();
  if (!(*a.flags & 1)) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = a.g;
  __shared__ float s_m[kSegWarps][kMaxG], s_l[kSegWarps][kMaxG];
  __shared__ float s_acc[kSegWarps][kMaxG][kD];
  for (int u = blockIdx.x; u < a.n_requests * a.H; u += gridDim.x) {
  const int b = u / a.H, h = u % a.H;
  const kvq_request& r = a.reqs[b];
  if (!attn_request_ok(a, r)) continue;  // the output is already NaN
  const int ns = r.n_sink, n = r.n_sink + r.n_tail;
  if (n == 0) continue;
  const float qscale = a.scale * kSegLog2e;
  float qv[kMaxG][4];
#pragma unroll
  for (int i = 0; i < kMaxG; ++i) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      qv[i][e] = i < g ? bf16_bits_to_f32(a.q[((long long)b * a.Hq + (long long)h * g + i) * kD + 4 * lane + e]) * qscale
                       : 0.0f;
  }
  float m[kMaxG], l[kMaxG], acc[kMaxG][4];
#pragma unroll
  for (int i = 0; i < kMaxG; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[i][e] = 0.0f;
  }
  for (int tok = warp; tok < n; tok += kSegWarps) {
    const bool sink = tok < ns;
    const long long row = ((long long)(sink ? tok : tok - ns) * a.H + h) * kD + 4 * lane;
    const uint2 kw = *reinterpret_cast<const uint2*>((sink ? r.sink_k : r.tail_k) + row);
    const uint2 vw = *reinterpret_cast<const uint2*>((sink ? r.sink_v : r.tail_v) + row);
    const float kf[4] = {__uint_as_float(kw.x << 16), __uint_as_float(kw.x & 0xFFFF0000u),
                         __uint_as_float(kw.y << 16), __uint_as_float(kw.y & 0xFFFF0000u)};
    const float vf[4] = {__uint_as_float(vw.x << 16), __uint_as_float(vw.x & 0xFFFF0000u),
                         __uint_as_float(vw.y << 16), __uint_as_float(vw.y & 0xFFFF0000u)};
#pragma unroll
    for (int i = 0; i < kMaxG; ++i) {
      if (i >= g) break;
      float s = qv[i][0] * kf[0] + qv[i][1] * kf[1] + qv[i][2] * kf[2] + qv[i][3] * kf[3];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      const float mn = fmaxf(m[i], s);
      const float al = m[i] == -INFINITY ? 0.0f : exp2f(m[i] - mn);
      const float p = exp2f(s - mn);
      l[i] = l[i] * al + p;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][e] = fmaf(p, vf[e], acc[i][e] * al);
      m[i] = mn;
    }
  }
#pragma unroll
  for (int i = 0; i < kMaxG; ++i) {
    if (lane == 0) {
      s_m[warp][i] = m[i];
      s_l[warp][i] = l[i];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) s_acc[warp][i][4 * lane + e] = acc[i][e];
  }
  __syncthreads();
  for (int i = 0; i < g; ++i) {  // thread = channel
    float ms = -INFINITY;
    for (int w = 0; w < kSegWarps; ++w) ms = fmaxf(ms, s_m[w][i]);
    float ls = 0.0f, cs = 0.0f;
    for (int w = 0; w < kSegWarps; ++w) {
      const float wt = s_m[w][i] == -INFINITY ? 0.0f : exp2f(s_m[w][i] - ms);
      ls += s_l[w][i] * wt;
      cs += s_acc[w][i][tid] * wt;
    }
    const long long oi = (long long)b * a.Hq + (long long)h * g + i;
    const float2 st = a.stats[oi];  // the packed part: max (log2 units), sum
    const bool packed = st.y > 0.0f && st.x != -INFINITY;
    const float M = packed ? fmaxf(st.x, ms) : ms;
    const float w0 = packed ? exp2f(st.x - M) : 0.0f;
    const float w1 = exp2f(ms - M);
    const float num = (packed ? a.out[oi * kD + tid] * (st.y * w0) : 0.0f) + cs * w1;
    const float den = (packed ? st.y * w0 : 0.0f) + ls * w1;
    a.out[oi * kD + tid] = num / den;
  }
  __syncthreads();  // the next unit reuses the shared arrays
  }
}

cudaError_t launch_segments(const AttnArgs& a, cudaStream_t stream) {
  if (a.n_requests == 0) return cudaSuccess;
  cudaError_t e = launch_dependent(segment_kernel, dim3(unit_grid(a)), dim3(32 * kSegWarps), 0, stream, a);
  count_launch();
  return e;
}

// ---------------------------------------------------------------- CUDA-core attention

// Softmax state is kept in the log2 domain: logits are scaled by
// scale*log2(e) and exponentials are exp2.
constexpr float kLog2e = 1.4426950408889634f;

struct SimtSmem {
  float q[kMaxG][kD];
  float khat[KVQ_TILE][kD];
  float vhat[KVQ_TILE][kD];
  float p[KVQ_TILE][kMaxG];
  int map[KVQ_MAX_LOOPS][KVQ_TILE];
  float m[kMaxG];
  float l[kMaxG];
  float alpha[kMaxG];
  Chain ck;
  Chain cv;
};

__device__ void simt_load_unit(const AttnArgs& a, SimtSmem& S, int b, int h) {
  const int tid = threadIdx.x;
  for (int k = tid; k < a.g * kD; k += blockDim.x) {
    int i = k / kD, d = k % kD;
    S.q[i][d] = bf16_bits_to_f32(a.q[((long long)b * a.Hq + (long long)h * a.g + i) * kD + d]) * (a.scale * kLog2e);
  }
  if (tid < kMaxG) {
    S.m[tid] = -INFINITY;
    S.l[tid] = 0.0f;
  }
  if (tid == 0) {
    const kvq_request& r = a.reqs[b];
    for (int kind = 0; kind < 2; ++kind) {
      Chain& C = kind == 0 ? S.ck : S.cv;
      C.depth = a.depth;
      C.kind = kind;
      C.n_tokens = r.n_tokens;
      C.n_heads = a.H;
      for (int j = 0; j < a.depth; ++j) planes_of(r, j, kind, C.loop[j]);
    }
  }
}

__device__ void simt_finish_unit(const AttnArgs& a, SimtSmem& S, float* acc, int b, int h, int u, bool whole) {
  const int tid = threadIdx.x;
  const int g = a.g;
  if (whole) {
    for (int k = tid, n = 0; k < g * kD; k += blockDim.x, ++n) {
      int i = k / kD, d = k % kD;
      a.out[((long long)b * a.Hq + (long long)h * g + i) * kD + d] = acc[n] / S.l[i];
    }
    if (tid < g) a.stats[(long long)b * a.Hq + (long long)h * g + tid] = make_float2(S.m[tid], S.l[tid]);
  } else {
    float* slot = a.partials + (size_t)(blockIdx.x + u) * kSlotFloats;
    if (tid < g) {
      slot[tid] = S.m[tid];
      slot[kMaxG + tid] = S.l[tid];
    }
    for (int k = tid, n = 0; k < g * kD; k += blockDim.x, ++n) {
      int i = k / kD, d = k % kD;
      slot[2 * kMaxG + i * kD + d] = acc[n];
    }
  }
}

__global__ void __launch_bounds__(256) attn_simt_kernel(AttnArgs a) {
  extern __shared__ __align__(16) uint8_t simt_smem[];
  SimtSmem& S = *reinterpret_cast<SimtSmem*>(simt_smem);
  const int tid = threadIdx.x;
  const int C = a.n_ctas;
  const long long W = a.prefix[a.n_requests];
  const long long s0 = cta_start(blockIdx.x, W, C), e0 = cta_start(blockIdx.x + 1, W, C);
  if (s0 >= e0) return;
  const int g = a.g;
  constexpr int kAccMax = kMaxG * kD / 256;  // pairs (head, channel) per thread
  float acc[kAccMax];

  int b = request_of(a.prefix, a.n_requests, s0);
  long long x = s0;
  while (x < e0) {
    // advance b to the request that owns tile x (skipping empty requests)
    while (a.prefix[b + 1] <= x) ++b;
    const kvq_request& r = a.reqs[b];
    const int T = r.n_tokens;
    const int nt = n_tiles_of(T);
    const long long rb = a.prefix[b];
    const int h = int((x - rb) / nt);
    const long long us = rb + (long long)h * nt, ue = us + nt;
    const int u = b * a.H + h;
    const long long xe = ue < e0 ? ue : e0;

    __syncthreads();
    simt_load_unit(a, S, b, h);
#pragma unroll
    for (int n = 0; n < kAccMax; ++n) acc[n] = 0.0f;
    __syncthreads();

    for (; x < xe; ++x) {
      const int k = int(x - us);
      const int t0 = k * KVQ_TILE;
      const int nvalid = min(KVQ_TILE, T - t0);
      // logical -> stored row for every loop
      for (int idx = tid; idx < a.depth * KVQ_TILE; idx += blockDim.x) {
        int j = idx / KVQ_TILE, tt = idx % KVQ_TILE;
        S.map[j][tt] = (S.ck.loop[j].sparse || tt >= nvalid) ? -1 : t0 + tt;
      }
      __syncthreads();
      for (int j = 1; j < a.depth; ++j) {
        const LoopPlanes& L = S.ck.loop[j];
        if (!L.sparse) continue;
        int c0 = __ldg(L.tile_dir + k), c1 = __ldg(L.tile_dir + k + 1);
        if (c0 < 0 || c1 > L.n_rows || c1 - c0 > KVQ_TILE || c0 > c1) {
          if (tid == 0) atomicOr(a.err, 4);
          continue;
        }
        for (int c = c0 + tid; c < c1; c += blockDim.x) {
          int tt = __ldg(L.active + c) - t0;
          if (tt >= 0 && tt < KVQ_TILE) S.map[j][tt] = c;
          else atomicOr(a.err, 4);
        }
      }
      __syncthreads();
      // FP32 decode of the chain (no BF16 rounding) for the tile's K and V rows
      for (int idx = tid; idx < KVQ_TILE * (kD / 4); idx += blockDim.x) {
        int tt = idx / (kD / 4), c0 = (idx % (kD / 4)) * 4;
        if (tt < nvalid) {
          int rows[KVQ_MAX_LOOPS];
          for (int j = 0; j < a.depth; ++j) rows[j] = S.map[j][tt];
          float kv[4], vv[4];
          chain4_f32(S.ck, a.depth, rows, t0 + tt, h, c0, kv);
          chain4_f32(S.cv, a.depth, rows, t0 + tt, h, c0, vv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            S.khat[tt][c0 + e] = kv[e];
            S.vhat[tt][c0 + e] = vv[e];
          }
        }
      }
      __syncthreads();
      // logits (log2 units)
      for (int idx = tid; idx < KVQ_TILE * g; idx += blockDim.x) {
        int tt = idx / g, i = idx % g;
        float sacc = -INFINITY;
        if (tt < nvalid && t0 + tt >= r.n_sink) {  // sink tokens are read from their BF16 copy instead
          sacc = 0.0f;
          for (int d = 0; d < kD; ++d) sacc = fmaf(S.q[i][d], S.khat[tt][d], sacc);
        }
        S.p[tt][i] = sacc;
      }
      __syncthreads();
      if (tid < g) {
        float mt = -INFINITY;
        for (int tt = 0; tt < nvalid; ++tt) mt = fmaxf(mt, S.p[tt][tid]);
        float mn = fmaxf(S.m[tid], mt);
        float al = (S.m[tid] == -INFINITY) ? 0.0f : exp2f(S.m[tid] - mn);
        float sum = 0.0f;
        for (int tt = 0; tt < KVQ_TILE; ++tt) {
          float p = (tt < nvalid && S.p[tt][tid] != -INFINITY) ? exp2f(S.p[tt][tid] - mn) : 0.0f;
          S.p[tt][tid] = p;
          sum += p;
        }
        S.alpha[tid] = al;
        S.l[tid] = S.l[tid] * al + sum;
        S.m[tid] = mn;
      }
      __syncthreads();
      {
        int n = 0;
        for (int kk = tid; kk < g * kD; kk += blockDim.x, ++n) {
          int i = kk / kD, d = kk % kD;
          float s = acc[n] * S.alpha[i];
          for (int tt = 0; tt < nvalid; ++tt) s = fmaf(S.p[tt][i], S.vhat[tt][d], s);
          acc[n] = s;
        }
      }
      __syncthreads();
    }
    simt_finish_unit(a, S, acc, b, h, u, us >= s0 && ue <= e0);
  }
}

cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t stream) {
  const int smem = int(sizeof(SimtSmem));
  static int configured = 0;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = 1;
  }
  attn_simt_kernel<<<a.n_ctas, 256, smem, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvq
