// kvq_sparse.cu — sparse decode attention over packed K/V (FlashLoop RFC,
// vllm-rlt issue #156, §3.2).
//
// At the reference loop the full attention is computed and, per query head,
// the keys S of largest probability are kept with their mass m, the full
// output O_ref and their contribution C_ref = sum_{t in S} p_t v_t; a later
// loop r attends over S only, at its own depth, and returns
//   O = O_ref - C_ref + m * softmax(q_r . K_r[S] / sqrt(d)) V_r[S].
// Historical K/V are read from the packed chain (decoded in FP32, as the
// dense reader does); the keys of S are gathered row by row.
//
// Kernels (ours):
//   sparse_logits_kernel  block = (request, KV head, 64-token tile): the FP32
//                         logits (log2 units) of every key for the g query heads
//   sparse_select_kernel  block = (request, query head): softmax max and sum,
//                         exact top-k by a radix select of up to four passes
//                         on order-preserving keys (ties: lower position), the
//                         selected indices in ascending order, m and C_ref
//   sparse_attn_kernel    block = (request, query head): the later loop
#include "kvq_attn_common.cuh"
#include "kvq_sparse.cuh"

namespace kvq {

namespace {

constexpr float kL2e = 1.4426950408889634f;

// The K or V chain of a request as the decode helpers read it.
__device__ void chain_of(const kvq_request& r, int kind, int depth, int H, Chain& C) {
  C.depth = depth;
  C.kind = kind;
  C.n_tokens = r.n_tokens;
  C.n_heads = H;
  for (int j = 0; j < depth; ++j) planes_of(r, j, kind, C.loop[j]);
}

// A request the sparse kernels accept: a consistent packed chain, no BF16
// segments, at most max_tokens keys.
__device__ __forceinline__ bool sparse_request_ok(const kvq_request& r, int depth, int max_tokens) {
  return request_ok(r, depth) && r.n_sink == 0 && r.n_tail == 0 && r.n_tokens <= max_tokens;
}

// Stored rows of token t in loops 0..depth-1 (-1: absent, inherit).
__device__ __forceinline__ void rows_of(const Chain& C, int depth, int t, int* rows) {
  for (int j = 0; j < depth; ++j) rows[j] = row_of(C.loop[j], t);
}

// Order-preserving unsigned key of a float (larger float, larger key).
__device__ __forceinline__ uint32_t okey(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

}  // namespace

// ---------------------------------------------------------------- logits

__global__ void __launch_bounds__(128) sparse_logits_kernel(SparseArgs a) {
  const int u = blockIdx.x, k = blockIdx.y;
  const int b = u / a.H, h = u % a.H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const kvq_request& r = a.reqs[b];
  if (!sparse_request_ok(r, a.depth, a.max_tokens)) return;
  const int T = r.n_tokens;
  const int t0 = k * KVQ_TILE;
  if (t0 >= T) return;
  const int g = a.g;
  __shared__ Chain C;
  __shared__ float qs[kMaxG][kD];
  if (threadIdx.x == 0) chain_of(r, KVQ_K, a.depth, a.H, C);
  for (int i = 0; i < g; ++i)
    qs[i][threadIdx.x] =
        bf16_bits_to_f32(a.q[((long long)b * a.Hq + (long long)h * g + i) * kD + threadIdx.x]) * (a.scale * kL2e);
  __syncthreads();
  const int nvalid = min(KVQ_TILE, T - t0);
  for (int tt = warp; tt < nvalid; tt += 4) {
    const int t = t0 + tt;
    int rows[KVQ_MAX_LOOPS];
    rows_of(C, a.depth, t, rows);
    float kv[4];
    chain4_f32(C, a.depth, rows, t, h, 4 * lane, kv);
    for (int i = 0; i < g; ++i) {
      float s = qs[i][4 * lane] * kv[0] + qs[i][4 * lane + 1] * kv[1] + qs[i][4 * lane + 2] * kv[2] +
                qs[i][4 * lane + 3] * kv[3];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (lane == 0) a.logits[((long long)b * a.Hq + (long long)h * g + i) * a.max_tokens + t] = s;
    }
  }
}

// ---------------------------------------------------------------- selection, m and C_ref

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
static_assert(kSelThreads == 256, "one histogram bin per thread");
// Requests of up to this many keys keep their order-preserving keys in shared
// memory for the selection's passes; longer ones re-read the logits.
constexpr int kSelStageMax = 12288;
// The first this many selected positions also go to shared memory, from which
// the C_ref gather reads them.
constexpr int kSelListMax = 1024;

// Block-wide exclusive scan of one flag per thread; returns the prefix and
// writes the total to *total (every thread).
__device__ __forceinline__ int block_scan(int flag, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned ball = __ballot_sync(0xffffffffu, flag);
  const int within = __popc(ball & ((1u << lane) - 1u));
  if (lane == 0) s_warp[warp] = __popc(ball);
  __syncthreads();
  int before = 0, sum = 0;
  for (int w = 0; w < kSelWarps; ++w) {
    const int c = s_warp[w];
    if (w < warp) before += c;
    sum += c;
  }
  __syncthreads();
  *total = sum;
  return before + within;
}

// The float of an order-preserving key.
__device__ __forceinline__ float okey_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The FP32 chain of V at a stored-row set over channels c0 .. c0 + 15 (c0 a
// multiple of 16: one V group, one NVFP4 block): the arithmetic of
// chain4_f32, with one 8-byte codes load and one parameter pair per loop. The
// decode min + scale * c is one FMA: scale * c is exact (an FP16 significand
// times a 4-bit code), so the FMA rounds once where chain4_f32 rounds the sum.
__device__ __forceinline__ void chain16_v_f32(const Chain& C, int depth, const int* rows, int h, int c0,
                                              float out[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) out[e] = 0.0f;
  for (int j = 0; j < depth; ++j) {
    const int row = rows[j];
    if (row < 0) continue;
    const LoopPlanes& L = C.loop[j];
    const long long rr = (long long)h * L.stride + row;
    const uint2 cw = __ldg(reinterpret_cast<const uint2*>(L.codes + rr * kRowBytes + c0 / 2));
    if (L.fmt == KVQ_FMT_NVFP4) {
      const float sb = nvfp4_block_scale(L, h, row, c0 / 16), st = nvfp4_tensor_scale(L);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float dq = nvfp4_dequant(((e < 8 ? cw.x : cw.y) >> (4 * (e & 7))) & 0xFu, sb, st);
        out[e] = (j == 0) ? dq : __fadd_rn(out[e], dq);
      }
      continue;
    }
    const long long pi = rr * (kD / kG) + c0 / kG;
    const float mn = f16_bits_to_f32(__ldg(L.mins + pi)), sc = f16_bits_to_f32(__ldg(L.scales + pi));
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t nib = ((e < 8 ? cw.x : cw.y) >> (4 * (e & 7))) & 0xFu;
      const float dq = __fmaf_rn(sc, __uint_as_float(nib | 0x4B000000u) - 8388608.0f, mn);
      out[e] = (j == 0) ? dq : __fadd_rn(out[e], dq);
    }
  }
}

// Block = (request, query head). The logits become order-preserving keys
// (staged in shared memory when the request fits); the K-th largest key comes
// from up to four radix passes over the key bytes, most significant first: a
// block histogram of the keys that share the prefix found so far (increments
// aggregated per warp and bin), then one warp finds the bin holding the K-th
// key by a suffix sum over its lanes. When that bin is taken whole the
// threshold is its lowest key and the passes stop early. Positions are then
// compacted in order (ties at the threshold: lower positions first), and C_ref
// gathers the selected V rows, four keys per warp at a time (eight lanes per
// key, sixteen channels per lane).
__global__ void __launch_bounds__(kSelThreads) sparse_select_kernel(SparseArgs a, int staged) {
  extern __shared__ uint32_t s_key[];  // [max_tokens] when staged
  const int bq = blockIdx.x;
  const int b = bq / a.Hq, hq = bq % a.Hq;
  const int h = hq / a.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const kvq_request& r = a.reqs[b];
  int32_t* sel = a.sel_idx + (long long)bq * a.n_select;
  float* cref = a.c_ref + (long long)bq * kD;
  const bool ok = sparse_request_ok(r, a.depth, a.max_tokens);
  const int T = ok ? r.n_tokens : 0;
  const int K = min(a.n_select, T);
  for (int i = K + tid; i < a.n_select; i += kSelThreads) sel[i] = -1;
  if (!ok) {
    if (tid == 0) {
      atomicOr(a.err, 1);
      a.mass[bq] = __int_as_float(0x7fc00000);
    }
    if (tid < kD) cref[tid] = __int_as_float(0x7fc00000);
    return;
  }
  if (K == 0) {
    if (tid == 0) a.mass[bq] = 0.0f;
    if (tid < kD) cref[tid] = 0.0f;
    return;
  }
  const float* s = a.logits + (long long)bq * a.max_tokens;
  __shared__ float s_red[kSelWarps];
  __shared__ int s_warp[kSelWarps];
  __shared__ unsigned s_hist[256];
  __shared__ unsigned s_prefix, s_need, s_whole;
  __shared__ Chain C;
  __shared__ float s_acc[kSelWarps][kD];
  __shared__ int s_sel[kSelListMax];
  auto key_at = [&](int t) -> uint32_t { return staged ? s_key[t] : okey(s[t]); };

  // softmax max (and the staged keys), then the sum (log2 units)
  float mx = -INFINITY;
  for (int t = tid; t < T; t += kSelThreads) {
    const float v = s[t];
    if (staged) s_key[t] = okey(v);
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) s_red[warp] = mx;
  if (tid == 0) {
    s_prefix = 0;
    s_need = unsigned(K);  // keys still to take at and below the current prefix
    s_whole = 0;
  }
  __syncthreads();
  float M = s_red[0];
  for (int w = 1; w < kSelWarps; ++w) M = fmaxf(M, s_red[w]);
  __syncthreads();
  float sum = 0.0f;
  for (int t = tid; t < T; t += kSelThreads) sum += exp2f(okey_value(key_at(t)) - M);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane == 0) s_red[warp] = sum;
  __syncthreads();
  float L = 0.0f;
  for (int w = 0; w < kSelWarps; ++w) L += s_red[w];

  // the threshold key
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    s_hist[tid] = 0;  // kSelThreads == 256 bins
    __syncthreads();
    const unsigned prefix = s_prefix;
    const unsigned hmask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
    // logits of one request crowd a few bins (the top byte is the sign and most
    // of the exponent): one shared atomic per warp and bin
    for (int base = 0; base < T; base += kSelThreads) {
      const int t = base + tid;
      const uint32_t key = t < T ? key_at(t) : 0u;
      const bool in = t < T && (key & hmask) == (prefix & hmask);
      if (__ballot_sync(0xffffffffu, in) != 0u) {
        const unsigned bin = (key >> shift) & 0xFFu;
        const unsigned peers = __match_any_sync(0xffffffffu, in ? bin : 256u + unsigned(lane));
        if (in && __ffs(peers) - 1 == lane) atomicAdd(&s_hist[bin], unsigned(__popc(peers)));
      }
    }
    __syncthreads();
    if (warp == 0) {  // lane l holds bins 8l .. 8l + 7; the suffix sums run from the top bin down
      const unsigned need = s_need;
      unsigned mine = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) mine += s_hist[8 * lane + k];
      unsigned suf = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned v = __shfl_down_sync(0xffffffffu, suf, off);
        if (lane + off < 32) suf += v;
      }
      const unsigned reach = __ballot_sync(0xffffffffu, suf >= need);  // lanes 0 .. l*
      const int ls = reach ? 31 - __clz(reach) : 0;
      if (lane == ls) {
        unsigned acc = suf - mine;  // keys in the bins above this lane's
        int bin = 8 * lane + 7;
        for (; bin > 8 * lane; --bin) {
          if (acc + s_hist[bin] >= need) break;
          acc += s_hist[bin];
        }
        s_prefix = prefix | (unsigned(bin) << shift);
        s_need = need - acc;  // keys to take equal to the prefix so far
        s_whole = (acc + s_hist[bin] == need) ? 1u : 0u;
      }
    }
    __syncthreads();
    if (s_whole) break;
  }
  const uint32_t tau = s_prefix;  // the K-th largest key, or the lowest key of a bin taken whole
  const unsigned take_eq = s_whole ? 0xFFFFFFFFu : s_need;  // keys equal to tau to take, lowest positions first

  // compaction in position order; m from the selected probabilities
  int written = 0, eq_seen = 0;
  float msum = 0.0f;
  for (int base = 0; base < T; base += kSelThreads) {
    const int t = base + tid;
    const uint32_t key = t < T ? key_at(t) : 0u;
    const int is_eq = (t < T && key == tau) ? 1 : 0;
    int eq_total = 0, eq_before = 0;  // keys equal to tau are counted only when some are left out
    if (take_eq != 0xFFFFFFFFu) eq_before = eq_seen + block_scan(is_eq, s_warp, &eq_total);
    const int take = (t < T) && (key > tau || (is_eq && unsigned(eq_before) < take_eq));
    int n_take = 0;
    const int pos = written + block_scan(take, s_warp, &n_take);
    if (take) {
      sel[pos] = t;
      if (pos < kSelListMax) s_sel[pos] = t;
      msum += exp2f(okey_value(key) - M);
    }
    written += n_take;
    eq_seen += eq_total;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) msum += __shfl_xor_sync(0xffffffffu, msum, off);
  if (lane == 0) s_red[warp] = msum;
  if (tid == 0) chain_of(r, KVQ_V, a.depth, a.H, C);
  __syncthreads();  // also orders the selected positions before their reads below
  if (tid == 0) {
    float ms = 0.0f;
    for (int w = 0; w < kSelWarps; ++w) ms += s_red[w];
    a.mass[bq] = ms / L;
  }

  // C_ref: the selected rows of V at the reference depth, weighted by p; a
  // warp takes four keys at a time, eight lanes per key
  const int ks = lane >> 3, sub = lane & 7;
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.0f;
  for (int i0 = 4 * warp; i0 < K; i0 += 4 * kSelWarps) {
    const int i = i0 + ks;
    if (i < K) {
      const int t = i < kSelListMax ? s_sel[i] : sel[i];
      int rows[KVQ_MAX_LOOPS];
      rows_of(C, a.depth, t, rows);
      float vv[16];
      chain16_v_f32(C, a.depth, rows, h, 16 * sub, vv);
      const float p = exp2f(okey_value(key_at(t)) - M) / L;
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = fmaf(p, vv[e], acc[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 8);
    acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
  }
  if (ks == 0) {
#pragma unroll
    for (int e = 0; e < 16; ++e) s_acc[warp][16 * sub + e] = acc[e];
  }
  __syncthreads();
  if (tid < kD) {
    float c = 0.0f;
    for (int w = 0; w < kSelWarps; ++w) c += s_acc[w][tid];
    cref[tid] = c;
  }
}

// ---------------------------------------------------------------- later loop

constexpr int kAttnWarps = 4;

__global__ void __launch_bounds__(32 * kAttnWarps) sparse_attn_kernel(SparseArgs a) {
  const int bq = blockIdx.x;
  const int b = bq / a.Hq, hq = bq % a.Hq;
  const int h = hq / a.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const kvq_request& r = a.reqs[b];
  float* out = a.out + (long long)bq * kD;
  const bool ok = sparse_request_ok(r, a.depth, a.max_tokens);
  if (!ok) {
    if (tid == 0) atomicOr(a.err, 1);
    out[tid] = __int_as_float(0x7fc00000);
    return;
  }
  const int K = min(a.n_select, r.n_tokens);
  const int32_t* sel = a.sel_idx + (long long)bq * a.n_select;
  __shared__ Chain CK, CV;
  __shared__ float qs[kD];
  __shared__ float s_m[kAttnWarps], s_l[kAttnWarps];
  __shared__ float s_acc[kAttnWarps][kD];
  if (tid == 0) {
    chain_of(r, KVQ_K, a.depth, a.H, CK);
    chain_of(r, KVQ_V, a.depth, a.H, CV);
  }
  qs[tid] = bf16_bits_to_f32(a.q[(long long)bq * kD + tid]) * (a.scale * kL2e);
  __syncthreads();
  float m = -INFINITY, l = 0.0f, acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  bool bad = false;
  // a warp takes 32 consecutive selected keys at a time: lane i resolves the
  // stored rows of key i (the searches run side by side), then the warp walks
  // the 32 keys with the rows passed by shuffles
  for (int base = 32 * warp; base < K; base += 32 * kAttnWarps) {
    const int nk = min(32, K - base);
    int my_t = lane < nk ? sel[base + lane] : -1;
    const bool my_bad = lane < nk && (my_t < 0 || my_t >= r.n_tokens);  // not a selection of this request
    if (my_bad) my_t = -1;
    bad |= __any_sync(0xffffffffu, my_bad);
    int my_rows[KVQ_MAX_LOOPS];
    for (int j = 0; j < a.depth; ++j) my_rows[j] = my_t >= 0 ? row_of(CK.loop[j], my_t) : -1;
    for (int kk = 0; kk < nk; ++kk) {
      const int t = __shfl_sync(0xffffffffu, my_t, kk);
      int rows[KVQ_MAX_LOOPS];
      for (int j = 0; j < a.depth; ++j) rows[j] = __shfl_sync(0xffffffffu, my_rows[j], kk);
      if (t < 0) continue;
      float kv[4], vv[4];
      chain4_f32(CK, a.depth, rows, t, h, 4 * lane, kv);
      chain4_f32(CV, a.depth, rows, t, h, 4 * lane, vv);
      float s = qs[4 * lane] * kv[0] + qs[4 * lane + 1] * kv[1] + qs[4 * lane + 2] * kv[2] + qs[4 * lane + 3] * kv[3];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      const float mn = fmaxf(m, s);
      const float al = m == -INFINITY ? 0.0f : exp2f(m - mn);
      const float p = exp2f(s - mn);
      l = l * al + p;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = fmaf(p, vv[e], acc[e] * al);
      m = mn;
    }
  }
  if (bad && lane == 0) atomicOr(a.err, 32);
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) s_acc[warp][4 * lane + e] = acc[e];
  __syncthreads();
  float M = -INFINITY;
  for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_m[w]);
  float Lt = 0.0f, c = 0.0f;
  for (int w = 0; w < kAttnWarps; ++w) {
    const float wgt = s_m[w] == -INFINITY ? 0.0f : exp2f(s_m[w] - M);
    Lt += s_l[w] * wgt;
    c += s_acc[w][tid] * wgt;
  }
  const float cnew = Lt > 0.0f ? c / Lt : 0.0f;
  out[tid] = a.o_ref[(long long)bq * kD + tid] - a.c_ref[(long long)bq * kD + tid] + a.mass[bq] * cnew;
}

// ---------------------------------------------------------------- later loop on the tensor-core kernel
//
// The selections become key masks, one bit per position and (request, query
// head), for the packed tensor-core attention, which drops the logits of the
// unselected keys; its normalised output is softmax(q K[S]^T) V[S] and its
// (max, sum) state tells an empty selection. The epilogue applies the
// correction O_ref - C_ref + m * that output.

// One thread per selection entry; the mask words were zeroed before.
__global__ void __launch_bounds__(256) sparse_mask_kernel(SparseArgs a) {
  const long long n = (long long)a.n_requests * a.Hq * a.n_select;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long bq = i / a.n_select;
    const int k = int(i - bq * a.n_select);
    const kvq_request& r = a.reqs[bq / a.Hq];
    const int T = r.n_tokens;
    if (T > a.max_tokens || k >= min(a.n_select, T)) continue;  // refused request, or past the count
    const int t = a.sel_idx[i];
    if (t < 0 || t >= T) {  // not a selection of this request
      atomicOr(a.err, 32);
      continue;
    }
    atomicOr(a.sel_mask + bq * a.mask_words + (t >> 5), 1u << (t & 31));
  }
}

__global__ void __launch_bounds__(kD) sparse_epilogue_kernel(SparseArgs a) {
  const int bq = blockIdx.x, d = threadIdx.x;
  const kvq_request& r = a.reqs[bq / a.Hq];
  float* out = a.out + (long long)bq * kD;
  if (!sparse_request_ok(r, a.depth, a.max_tokens)) {
    if (d == 0) atomicOr(a.err, 1);
    out[d] = __int_as_float(0x7fc00000);
    return;
  }
  if (a.refuse_nvfp4) {  // refused by the attention's plan (bit 64): its softmax state was never written
    for (int j = 0; j < a.depth; ++j)
      if (r.loop[j].flags & (KVQ_LOOP_K_NVFP4 | KVQ_LOOP_V_NVFP4)) {
        out[d] = __int_as_float(0x7fc00000);
        return;
      }
  }
  const float cnew = a.stats[bq].y > 0.0f ? out[d] : 0.0f;  // an empty selection contributes nothing
  out[d] = a.o_ref[(long long)bq * kD + d] - a.c_ref[(long long)bq * kD + d] + a.mass[bq] * cnew;
}

cudaError_t launch_sparse_mask(const SparseArgs& a, cudaStream_t stream) {
  const long long n = (long long)a.n_requests * a.Hq * a.n_select;
  if (n == 0) return cudaSuccess;
  const long long blocks = (n + 255) / 256;
  sparse_mask_kernel<<<int(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_sparse_epilogue(const SparseArgs& a, cudaStream_t stream) {
  if (a.n_requests == 0) return cudaSuccess;
  sparse_epilogue_kernel<<<a.n_requests * a.Hq, kD, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_sparse_select_path(const SparseArgs& a, cudaStream_t stream) {
  if (a.n_requests == 0) return cudaSuccess;
  const int tiles = (a.max_tokens + KVQ_TILE - 1) / KVQ_TILE;
  if (tiles > 0) {
    sparse_logits_kernel<<<dim3(a.n_requests * a.H, tiles), 128, 0, stream>>>(a);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_sparse_select(a, stream);
}

cudaError_t launch_sparse_select(const SparseArgs& a, cudaStream_t stream) {
  if (a.n_requests == 0) return cudaSuccess;
  const int staged = a.max_tokens <= kSelStageMax ? 1 : 0;
  const size_t smem = staged ? size_t(a.max_tokens) * 4 : 0;
  static bool configured = false;
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(sparse_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kSelStageMax * 4);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  sparse_select_kernel<<<a.n_requests * a.Hq, kSelThreads, smem, stream>>>(a, staged);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_sparse_attn(const SparseArgs& a, cudaStream_t stream) {
  if (a.n_requests == 0) return cudaSuccess;
  sparse_attn_kernel<<<a.n_requests * a.Hq, 32 * kAttnWarps, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvq
