// kvq_attn_mma.cu — tensor-core decode attention over packed K/V.
//
// FlashLoop RFC (vllm-rlt issue #156) §3.2: historical K/V are read at the
// requested depth and reconstructed if compressed, scores scaled by
// 1/sqrt(head_dim); §3.3: readers consume the packed base/residual tiles
// directly during QK/PV instead of a BF16 shadow cache; §5: FP32 mass and
// accumulation. The dequantiser is the affine INT4 group code of §3.3
// (decode = min + scale * code).
//
// Design (ours). One CTA per SM runs over a contiguous range of 64-token tiles
// of the flat (request, KV head, tile) work list (kvq_attn_common.cuh).
//   producer warp   one lane issues 1-D bulk TMA copies (cp.async.bulk with
//                   mbarrier transaction counts) of each tile's packed planes —
//                   per loop: K and V codes, K and V min/scale planes, and for
//                   a sparse loop its index slice — into one of kStages stages.
//   8 consumer warps fold the dequantisation into the contractions, since min
//                   and scale are constant along each contraction:
//       S[t, h]  = sum_j [ sum_d c_j[t,d] * (q[h,d] * sK_j[d]) + sum_d q[h,d] * mK_j[d] ]
//       O[h, d]  = sum_j [ sum_t c_j[t,d] * (p[t,h] * sV_j[t]) + sum_t p[t,h] * mV_j[t] ]
//                   Codes are unpacked to exact FP16 integers in registers and
//                   fed to mma.sync m16n8k16 (FP32 accumulate). q (BF16) is
//                   exact in FP16; q*sK is carried exactly as the sum of two
//                   FP16 terms (hi = RN16(q*sK), lo = RN16(q*sK - hi)), so the
//                   logits are exact up to FP32 accumulation. QK^T runs with
//                   tokens as M and the 8 query heads of a KV head as N, PV
//                   with channels as M. Sparse loops are processed over their
//                   compact rows only; their logits are gathered back to
//                   logical tokens through a 64-bit presence mask per tile.
//                   The K min terms of all (loop, group) pairs come from one
//                   small MMA; the V min terms are FP32 sums.
// Softmax is online over tiles in the log2 domain, FP32 throughout.
#include <cuda_fp16.h>

#include "kvq_attn_common.cuh"

namespace kvq {
namespace mma_attn {

constexpr int kLoops = 4;            // depth handled by this kernel
constexpr int kStages = 3;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + producer warp
constexpr int kMaxPairs = 2 * kLoops;       // (loop, K group) pairs of one tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitNs = 2000000000LL;  // bounded waits: 2 s, then flag and leave

// Per-loop description of a staged tile.
struct LoopMeta {
  int32_t nrows;   // stored rows in this tile (logical rows for dense, compact rows for sparse)
  int32_t c0;      // first stored row (stream row index)
  int32_t g0;      // K group of row c0
  int32_t ngrp;    // K groups spanned (1 or 2; 0 if no rows)
  int32_t vrem;    // half offset of the first V param inside the staged V param chunk
  int32_t irem;    // int offset of the first index inside the staged index chunk
  int32_t sparse;
  int32_t pad;
};

struct TileMeta {
  int32_t unit;    // b*H + h
  int32_t b, h;
  int32_t t0, nvalid;
  int32_t whole;   // this CTA covers the unit's whole tile range
  int32_t last_of_unit;
  int32_t pad;
  LoopMeta loop[kLoops];
};

struct __align__(128) Stage {
  uint8_t kc[kLoops][KVQ_TILE * kRowBytes];
  uint8_t vc[kLoops][KVQ_TILE * kRowBytes];
  uint16_t kmin[kLoops][2 * kD];
  uint16_t ksc[kLoops][2 * kD];
  uint16_t vmin[kLoops][144];  // 64 rows x 2 groups + 16 B rounding slack
  uint16_t vsc[kLoops][144];
  int32_t idx[kLoops][80];     // 64 indices + rounding slack
  TileMeta meta;
};

struct Smem {
  Stage st[kStages];
  // Q' = q * sK per (pair, head) as FP16 hi and lo terms, fragment order: head
  // stride 160 halves (320 B), then [word i][chunk q][8 channels in the order
  // 0,4,1,5,2,6,3,7].
  __half qp[kMaxPairs][2][8 * 160];
  float kbias[kMaxPairs][8];                // sum_d q * mK per (pair, head)
  float s[kLoops][KVQ_TILE][8];             // per-loop logits (stream rows), log2 units
  // P' = p * sV per (loop, V group), FP16, fragment order [k-step][head][16].
  __half pp[kLoops][2][4][8][16];
  __half q16[8][kD];                        // query of the current unit (BF16 values, exact in FP16)
  float fin[4][kD][8];                      // end-of-unit sum of the row-quarter PV partials
  unsigned long long mask[kLoops];          // presence of logical tokens in a sparse loop
  float red[kConsumerWarps][8];
  float alpha[8];
  float lsum[kConsumerWarps][8];
  float vbs[kConsumerWarps][8][2];
  float vbias[8][2];
  float l_tot[8];
  int32_t pair_j[kMaxPairs], pair_g[kMaxPairs];
  int32_t npairs;
  unsigned long long full[kStages];
  unsigned long long empty[kStages];
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of `bar`; gives up after kWaitNs (returns false).
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitNs) return false;
  }
  return true;
}

// Adds `bytes` to the barrier's expected transaction count, then starts the copy.
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, unsigned long long* bar) {
  mbar_expect_tx(bar, bytes);
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t m, uint32_t o) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(r) : "r"(a), "r"(m), "r"(o));
  return r;
}

__device__ __forceinline__ uint32_t h2_sub1024(uint32_t x) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&x), __half2(__float2half_rn(1024.f), __float2half_rn(1024.f)));
  return *reinterpret_cast<uint32_t*>(&r);
}

// (1024 + 16c) / 16 - 64 = c
__device__ __forceinline__ uint32_t h2_hi_nibble(uint32_t x) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&x), __half2(__float2half_rn(0.0625f), __float2half_rn(0.0625f)),
                      __half2(__float2half_rn(-64.f), __float2half_rn(-64.f)));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Codes of a 32-bit word w (nibbles n0..n7, n0 = lowest channel) as exact FP16 pairs:
// r[0] = {n0, n4}, r[1] = {n1, n5}, r[2] = {n2, n6}, r[3] = {n3, n7}.
__device__ __forceinline__ void unpack8(uint32_t w, uint32_t r[4]) {
  const uint32_t w8 = w >> 8;
  r[0] = h2_sub1024(lop3_and_or(w, 0x000F000Fu, 0x64006400u));
  r[1] = h2_hi_nibble(lop3_and_or(w, 0x00F000F0u, 0x64006400u));
  r[2] = h2_sub1024(lop3_and_or(w8, 0x000F000Fu, 0x64006400u));
  r[3] = h2_hi_nibble(lop3_and_or(w8, 0x00F000F0u, 0x64006400u));
}

__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ int popc64(unsigned long long x) { return __popcll(x); }

// ---------------------------------------------------------------- producer

struct UnitPtrs {
  int T;
  int nrows[kLoops];
  const int32_t* active[kLoops];
  const int32_t* dir[kLoops];
  const uint8_t* kc[kLoops];
  const uint16_t* kmin[kLoops];
  const uint16_t* ksc[kLoops];
  const uint8_t* vc[kLoops];
  const uint16_t* vmin[kLoops];
  const uint16_t* vsc[kLoops];
};

__device__ void producer(const AttnArgs& a, Smem& S, long long s0, long long e0) {
  const long long W = a.prefix[a.n_requests];
  const int C = a.n_ctas;
  int b = request_of(a.prefix, a.n_requests, s0);
  int cur_unit = -1;
  UnitPtrs U;
  long long it = 0;
  for (long long x = s0; x < e0; ++x, ++it) {
    const int s = int(it % kStages);
    const uint32_t ph = uint32_t((it / kStages) & 1);
    if (it >= kStages && !mbar_wait(&S.empty[s], ph ^ 1u)) {
      atomicOr(a.err, 8);
      return;
    }
    while (a.prefix[b + 1] <= x) ++b;
    const kvq_request& R = a.reqs[b];
    const int T = R.n_tokens;
    const int nt = n_tiles_of(T);
    const long long rb = a.prefix[b];
    const int h = int((x - rb) / nt);
    const int k = int((x - rb) % nt);
    const int unit = b * a.H + h;
    if (unit != cur_unit) {
      cur_unit = unit;
      U.T = T;
      for (int j = 0; j < a.depth; ++j) {
        const kvq_loop_ref& L = R.loop[j];
        U.nrows[j] = L.n_rows;
        U.active[j] = L.active_idx;
        U.dir[j] = L.tile_dir;
        U.kc[j] = L.k_codes;
        U.kmin[j] = L.k_mins;
        U.ksc[j] = L.k_scales;
        U.vc[j] = L.v_codes;
        U.vmin[j] = L.v_mins;
        U.vsc[j] = L.v_scales;
      }
    }
    Stage& st = S.st[s];
    TileMeta& M = st.meta;
    M.unit = unit;
    M.b = b;
    M.h = h;
    M.t0 = k * KVQ_TILE;
    M.nvalid = min(KVQ_TILE, T - M.t0);
    const long long us = rb + (long long)h * nt, ue = us + nt;
    M.whole = (us >= s0 && ue <= e0) ? 1 : 0;
    M.last_of_unit = (x == ue - 1 || x == e0 - 1) ? 1 : 0;
    (void)W;
    (void)C;
    // rows of every loop
    int c0s[kLoops], c1s[kLoops];
    for (int j = 0; j < a.depth; ++j) {
      if (U.active[j] == nullptr) {
        c0s[j] = M.t0;
        c1s[j] = M.t0 + M.nvalid;
      } else {
        c0s[j] = __ldg(U.dir[j] + k);
        c1s[j] = __ldg(U.dir[j] + k + 1);
      }
    }
    uint32_t bytes = 0;
    for (int j = 0; j < a.depth; ++j) {
      int c0 = c0s[j], c1 = c1s[j];
      LoopMeta& LM = M.loop[j];
      LM.sparse = U.active[j] != nullptr;
      if (c0 < 0 || c1 > U.nrows[j] || c0 > c1 || c1 - c0 > KVQ_TILE) {
        atomicOr(a.err, 4);
        c0 = c1 = 0;
      }
      const int n = c1 - c0;
      LM.nrows = n;
      LM.c0 = c0;
      LM.g0 = c0 / kG;
      LM.ngrp = n > 0 ? (c1 - 1) / kG - c0 / kG + 1 : 0;
      LM.vrem = 0;
      LM.irem = 0;
      if (n == 0) continue;
      const int nr = U.nrows[j];
      // codes: n rows x 64 B, contiguous in the head-major plane
      bulk_copy(st.kc[j], U.kc[j] + ((long long)h * nr + c0) * kRowBytes, n * kRowBytes, &S.full[s]);
      bulk_copy(st.vc[j], U.vc[j] + ((long long)h * nr + c0) * kRowBytes, n * kRowBytes, &S.full[s]);
      bytes += 2 * n * kRowBytes;
      // K params: the spanned groups, 256 B per group and plane
      const int ng = (nr + kG - 1) / kG;
      const uint16_t* km = U.kmin[j] + ((long long)h * ng + LM.g0) * kD;
      const uint16_t* ks = U.ksc[j] + ((long long)h * ng + LM.g0) * kD;
      bulk_copy(st.kmin[j], km, LM.ngrp * kD * 2, &S.full[s]);
      bulk_copy(st.ksc[j], ks, LM.ngrp * kD * 2, &S.full[s]);
      bytes += 2 * LM.ngrp * kD * 2;
      // V params: 4 B per row and plane, copied in 16-byte units (the planes are
      // allocated to a 16-byte multiple, so the rounded range stays inside)
      {
        const long long off = ((long long)h * nr + c0) * 4;  // bytes
        const long long lo = off & ~15LL;
        const long long hi = (off + (long long)n * 4 + 15) & ~15LL;
        const uint32_t nb = uint32_t(hi - lo);
        bulk_copy(st.vmin[j], reinterpret_cast<const uint8_t*>(U.vmin[j]) + lo, nb, &S.full[s]);
        bulk_copy(st.vsc[j], reinterpret_cast<const uint8_t*>(U.vsc[j]) + lo, nb, &S.full[s]);
        bytes += 2 * nb;
        LM.vrem = int((off - lo) / 2);
      }
      if (LM.sparse) {
        const long long off = (long long)c0 * 4;
        const long long lo = off & ~15LL;
        const long long hi = (off + (long long)n * 4 + 15) & ~15LL;
        const uint32_t nb = uint32_t(hi - lo);
        bulk_copy(st.idx[j], reinterpret_cast<const uint8_t*>(U.active[j]) + lo, nb, &S.full[s]);
        bytes += nb;
        LM.irem = int((off - lo) / 4);
      }
    }
    // The single expected arrival: releases the metadata written above; the phase
    // completes once every copy has delivered its bytes.
    (void)bytes;
    mbar_arrive(&S.full[s]);
  }
}

// ---------------------------------------------------------------- consumers

struct UnitState {
  float m;       // running max of this thread's head (log2 units)
  float l;       // partial sum of exp2 for this thread's (head, tokens)
  float vb[2];   // partial V-min terms per V group
  float acc[4][4];  // PV accumulators: 4 channel m-tiles x (2 rows x 2 heads)
};

__device__ void load_unit_query(const AttnArgs& a, Smem& S, int b, int h) {
  const int tid = threadIdx.x;
  for (int i = tid; i < 8 * kD; i += kConsumers) {
    const int hh = i / kD, d = i % kD;
    float v = 0.0f;
    if (hh < a.g) v = bf16_bits_to_f32(a.q[((long long)b * a.Hq + (long long)h * a.g + hh) * kD + d]);
    S.q16[hh][d] = __float2half_rn(v);  // exact: a BF16 value in the FP16 range
  }
}

// Writes the unit's result: output rows (whole unit) or a partial slot.
struct UnitInfo {
  int unit, b, h, whole;
};

__device__ void finish_unit(const AttnArgs& a, Smem& S, UnitState& U, const UnitInfo& M, int warp, int lane) {
  const int tid = threadIdx.x;
  const int hme = tid & 7;
  // l and V-min terms: reduce over the threads of the same head
  float l = U.l, v0 = U.vb[0], v1 = U.vb[1];
#pragma unroll
  for (int off = 8; off < 32; off <<= 1) {
    l += __shfl_xor_sync(0xffffffffu, l, off);
    v0 += __shfl_xor_sync(0xffffffffu, v0, off);
    v1 += __shfl_xor_sync(0xffffffffu, v1, off);
  }
  if (lane < 8) {
    S.lsum[warp][lane] = l;
    S.vbs[warp][lane][0] = v0;
    S.vbs[warp][lane][1] = v1;
  }
  // PV partials of this warp: channel group grp, row quarter rq
  const int grp = warp >> 2, rq = warp & 3;
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
    const int ch_lo = 64 * grp + 8 * g + 2 * mt;
    S.fin[rq][ch_lo][2 * q] = U.acc[mt][0];
    S.fin[rq][ch_lo][2 * q + 1] = U.acc[mt][1];
    S.fin[rq][ch_lo + 1][2 * q] = U.acc[mt][2];
    S.fin[rq][ch_lo + 1][2 * q + 1] = U.acc[mt][3];
  }
  consumer_sync();
  if (tid < 8) {
    float lt = 0.f, b0 = 0.f, b1 = 0.f;
    for (int w = 0; w < kConsumerWarps; ++w) {
      lt += S.lsum[w][tid];
      b0 += S.vbs[w][tid][0];
      b1 += S.vbs[w][tid][1];
    }
    S.l_tot[tid] = lt;
    S.vbias[tid][0] = b0;
    S.vbias[tid][1] = b1;
  }
  consumer_sync();
  const int g_q = a.g;
  if (M.whole) {
    for (int i = tid; i < g_q * kD; i += kConsumers) {
      const int hh = i / kD, d = i % kD;
      float o = S.fin[0][d][hh] + S.fin[1][d][hh] + S.fin[2][d][hh] + S.fin[3][d][hh] + S.vbias[hh][d >> 6];
      a.out[((long long)M.b * a.Hq + (long long)M.h * g_q + hh) * kD + d] = o / S.l_tot[hh];
    }
  } else {
    float* slot = a.partials + (size_t)(blockIdx.x + M.unit) * kSlotFloats;
    if (tid < g_q) {
      slot[tid] = U.m;  // every thread tracks the max of head tid & 7; thread tid has head tid
      slot[kMaxG + tid] = S.l_tot[tid];
    }
    for (int i = tid; i < g_q * kD; i += kConsumers) {
      const int hh = i / kD, d = i % kD;
      slot[2 * kMaxG + hh * kD + d] =
          S.fin[0][d][hh] + S.fin[1][d][hh] + S.fin[2][d][hh] + S.fin[3][d][hh] + S.vbias[hh][d >> 6];
    }
  }
  (void)hme;
  consumer_sync();
}

__device__ void consumer(const AttnArgs& a, Smem& S, long long s0, long long e0) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int hme = tid & 7;       // head of this thread in the softmax phase
  const int gq = a.g;
  UnitState U;
  int cur_unit = -1;
  UnitInfo Mprev = {-1, 0, 0, 0};
  long long it = 0;
  // Q' task of this thread: pair offset, head, channel chunk
  const int qt_pair = tid >> 7, qt_h = (tid >> 4) & 7, qt_chunk = tid & 15;
  uint32_t qreg[4];  // FP16 pairs of q in the order (0,4),(1,5),(2,6),(3,7) of the chunk

  for (long long x = s0; x < e0; ++x, ++it) {
    const int s = int(it % kStages);
    const uint32_t ph = uint32_t((it / kStages) & 1);
    if (!mbar_wait(&S.full[s], ph)) {
      if (lane == 0) atomicOr(a.err, 8);
      return;
    }
    Stage& st = S.st[s];
    const TileMeta& M = st.meta;
    if (M.unit != cur_unit) {
      if (cur_unit >= 0) finish_unit(a, S, U, Mprev, warp, lane);
      cur_unit = M.unit;
      U.m = -INFINITY;
      U.l = 0.f;
      U.vb[0] = U.vb[1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) U.acc[mt][e] = 0.f;
      load_unit_query(a, S, M.b, M.h);
      consumer_sync();
      {
        const __half* qp = &S.q16[qt_h][8 * qt_chunk];
        const __half o[8] = {qp[0], qp[4], qp[1], qp[5], qp[2], qp[6], qp[3], qp[7]};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __half2 hv = __halves2half2(o[2 * e], o[2 * e + 1]);
          qreg[e] = *reinterpret_cast<uint32_t*>(&hv);
        }
      }
    }
    Mprev.unit = M.unit;
    Mprev.b = M.b;
    Mprev.h = M.h;
    Mprev.whole = M.whole;
    const int depth = a.depth;

    // ---- prep: sparse presence masks, (loop, group) pairs, Q' and the K-min terms
    if (warp < depth && M.loop[warp].sparse) {
      const LoopMeta& LM = M.loop[warp];
      unsigned long long bits = 0;
      for (int i = lane; i < LM.nrows; i += 32) {
        const int u = st.idx[warp][LM.irem + i] - M.t0;
        if (u >= 0 && u < KVQ_TILE) bits |= 1ull << u;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, off);
      if (lane == 0) S.mask[warp] = bits;
    }
    if (tid == 0) {
      int np = 0;
      for (int j = 0; j < depth; ++j)
        for (int G = 0; G < M.loop[j].ngrp; ++G) {
          S.pair_j[np] = j;
          S.pair_g[np] = G;
          ++np;
        }
      S.npairs = np;
    }
    consumer_sync();
    const int npairs = S.npairs;
    for (int p = qt_pair; p < npairs; p += kConsumers / 128) {
      const int j = S.pair_j[p], G = S.pair_g[p];
      const uint4 sv = *reinterpret_cast<const uint4*>(&st.ksc[j][G * kD + 8 * qt_chunk]);
      // scales in the order (0,4),(1,5),(2,6),(3,7)
      const uint32_t s04 = __byte_perm(sv.x, sv.z, 0x5410), s15 = __byte_perm(sv.x, sv.z, 0x7632);
      const uint32_t s26 = __byte_perm(sv.y, sv.w, 0x5410), s37 = __byte_perm(sv.y, sv.w, 0x7632);
      const uint32_t sp[4] = {s04, s15, s26, s37};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __half2 qv = *reinterpret_cast<const __half2*>(&qreg[e]);
        const __half2 sv2 = *reinterpret_cast<const __half2*>(&sp[e]);
        const __half2 h2 = __hmul2(qv, sv2);                 // RN16(q * s)
        const __half2 l2 = __hfma2(qv, sv2, __hneg2(h2));   // RN16(q * s - hi), exact here
        hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
        lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
      }
      // chunk c covers channels 8c..8c+7 = 32q' + 8i': store at [head][i'][q']
      const int qq = qt_chunk >> 2, ii = qt_chunk & 3;
      *reinterpret_cast<uint4*>(&S.qp[p][0][qt_h * 160 + ii * 32 + qq * 8]) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(&S.qp[p][1][qt_h * 160 + ii * 32 + qq * 8]) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    // K-min terms of all pairs in one MMA chain: rows = pairs, K = channels, N = heads
    if (warp == kConsumerWarps - 1) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t av[4] = {0u, 0u, 0u, 0u};
        if (g < npairs) {
          const uint16_t* mrow = &st.kmin[S.pair_j[g]][S.pair_g[g] * kD + 16 * kk];
          av[0] = *reinterpret_cast<const uint32_t*>(mrow + 2 * q);
          av[2] = *reinterpret_cast<const uint32_t*>(mrow + 2 * q + 8);
        }
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&S.q16[g][16 * kk + 2 * q]);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&S.q16[g][16 * kk + 2 * q + 8]);
        mma16816(c, av, b0, b1);
      }
      if (g < npairs) {
        S.kbias[g][2 * q] = c[0];
        S.kbias[g][2 * q + 1] = c[1];
      }
    }
    consumer_sync();

    // ---- QK^T over the stored rows of every loop: item = (loop, 16-row m-tile)
    {
      int item = 0;
      int pbase = 0;
      for (int j = 0; j < depth; ++j) {
        const LoopMeta& LM = M.loop[j];
        const int nmt = (LM.nrows + 15) >> 4;
        for (int mt = 0; mt < nmt; ++mt, ++item) {
          if ((item % kConsumerWarps) != warp) continue;
          const int r0 = 16 * mt + g, r1 = r0 + 8;
          // K group of each row (relative to the tile's first group)
          const int ga = (LM.c0 + 16 * mt) / kG - LM.g0;
          const int gb = (LM.c0 + 16 * mt + 15) / kG - LM.g0;
          const bool split = ga != gb && gb < LM.ngrp;
          float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
          const uint4 wa = *reinterpret_cast<const uint4*>(&st.kc[j][r0 * kRowBytes + 16 * q]);
          const uint4 wb = *reinterpret_cast<const uint4*>(&st.kc[j][r1 * kRowBytes + 16 * q]);
          const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w}, wB[4] = {wb.x, wb.y, wb.z, wb.w};
          const __half* qpa = &S.qp[pbase + ga][0][g * 160 + q * 8];
          const __half* qpb = &S.qp[pbase + (split ? gb : ga)][0][g * 160 + q * 8];
          constexpr int kLo = 8 * 160;  // offset of the lo terms
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t ua[4], ub[4];
            unpack8(wA[i], ua);
            unpack8(wB[i], ub);
            const uint32_t A0[4] = {ua[0], ub[0], ua[1], ub[1]};
            const uint32_t A1[4] = {ua[2], ub[2], ua[3], ub[3]};
            const uint4 bh = *reinterpret_cast<const uint4*>(qpa + i * 32);
            const uint4 bl = *reinterpret_cast<const uint4*>(qpa + kLo + i * 32);
            mma16816(c0, A0, bh.x, bh.y);
            mma16816(c0, A1, bh.z, bh.w);
            mma16816(c0, A0, bl.x, bl.y);
            mma16816(c0, A1, bl.z, bl.w);
            if (split) {
              const uint4 bh2 = *reinterpret_cast<const uint4*>(qpb + i * 32);
              const uint4 bl2 = *reinterpret_cast<const uint4*>(qpb + kLo + i * 32);
              mma16816(c1, A0, bh2.x, bh2.y);
              mma16816(c1, A1, bh2.z, bh2.w);
              mma16816(c1, A0, bl2.x, bl2.y);
              mma16816(c1, A1, bl2.z, bl2.w);
            }
          }
          // rows r0 / r1 of this m-tile: pick the accumulator of their K group, add its min term
          const int gr0 = (LM.c0 + r0) / kG - LM.g0;
          const int gr1 = (LM.c0 + r1) / kG - LM.g0;
          const float* e0v = (split && gr0 != ga) ? c1 : c0;
          const float* e1v = (split && gr1 != ga) ? c1 : c0;
          const int p0 = pbase + min(gr0, LM.ngrp - 1), p1 = pbase + min(gr1, LM.ngrp - 1);
          *reinterpret_cast<float2*>(&S.s[j][r0][2 * q]) =
              make_float2(e0v[0] + S.kbias[p0][2 * q], e0v[1] + S.kbias[p0][2 * q + 1]);
          *reinterpret_cast<float2*>(&S.s[j][r1][2 * q]) =
              make_float2(e1v[2] + S.kbias[p1][2 * q], e1v[3] + S.kbias[p1][2 * q + 1]);
        }
        pbase += LM.ngrp;
      }
    }
    consumer_sync();

    // ---- softmax over the tile (online, log2 units) and P' = p * sV
    {
      // logits of this thread's tokens tt = tid/8 and tid/8 + 32 for head hme,
      // scaled into log2 units
      const float lsc = a.scale * kLog2e;
      float sv[2];
      int rows[2][kLoops];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int tt = (tid >> 3) + 32 * u;
        float acc = -INFINITY;
        if (tt < M.nvalid && hme < gq) {
          acc = 0.f;
          for (int j = 0; j < depth; ++j) {
            const LoopMeta& LM = M.loop[j];
            int row = tt;
            if (LM.sparse) {
              const unsigned long long mk = S.mask[j];
              row = ((mk >> tt) & 1ull) ? popc64(mk & ((1ull << tt) - 1ull)) : -1;
            }
            rows[u][j] = row;
            if (row >= 0) acc += S.s[j][row][hme];
          }
          acc *= lsc;
        } else {
          for (int j = 0; j < depth; ++j) rows[u][j] = -1;
        }
        sv[u] = acc;
      }
      float mloc = fmaxf(sv[0], sv[1]);
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 8));
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 16));
      if (lane < 8) S.red[warp][lane] = mloc;
      consumer_sync();
      float mt = S.red[0][hme];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) mt = fmaxf(mt, S.red[w][hme]);
      const float mnew = fmaxf(U.m, mt);
      const float alpha = (U.m == -INFINITY) ? 0.f : exp2f(U.m - mnew);
      U.m = mnew;
      if (tid < 8) S.alpha[tid] = alpha;
      U.l *= alpha;
      U.vb[0] *= alpha;
      U.vb[1] *= alpha;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int tt = (tid >> 3) + 32 * u;
        const float p = (sv[u] == -INFINITY) ? 0.f : exp2f(sv[u] - mnew);
        U.l += p;
        const __half2 p2 = __floats2half2_rn(p, p);
        for (int j = 0; j < depth; ++j) {
          const LoopMeta& LM = M.loop[j];
          const int row = LM.sparse ? rows[u][j] : tt;
          if (row < 0 || hme >= gq) continue;
          if (LM.sparse && row >= LM.nrows) continue;
          const int vi = LM.vrem + 2 * row;
          const __half2 sc2 = *reinterpret_cast<const __half2*>(&st.vsc[j][vi]);
          const __half2 pv = (p != 0.f) ? __hmul2(p2, sc2) : __float2half2_rn(0.f);
          const int ks = row >> 4, rr = row & 15;
          const int pos = 4 * (rr & 3) + (rr >> 2);
          S.pp[j][0][ks][hme][pos] = __low2half(pv);
          S.pp[j][1][ks][hme][pos] = __high2half(pv);
          if (p != 0.f) {
            const float2 mv = __half22float2(*reinterpret_cast<const __half2*>(&st.vmin[j][vi]));
            U.vb[0] = fmaf(p, mv.x, U.vb[0]);
            U.vb[1] = fmaf(p, mv.y, U.vb[1]);
          }
        }
      }
      // sparse loops: zero P' of the compact rows past nrows inside the last k-step
      for (int j = 0; j < depth; ++j) {
        const LoopMeta& LM = M.loop[j];
        if (!LM.sparse) continue;
        const int pad_end = (LM.nrows + 15) & ~15;
        for (int i = tid; i < (pad_end - LM.nrows) * 8; i += kConsumers) {
          const int row = LM.nrows + i / 8, hh = i % 8;
          const int ks = row >> 4, rr = row & 15;
          const int pos = 4 * (rr & 3) + (rr >> 2);
          S.pp[j][0][ks][hh][pos] = __float2half_rn(0.f);
          S.pp[j][1][ks][hh][pos] = __float2half_rn(0.f);
        }
      }
    }
    consumer_sync();

    // ---- PV: warp = (V group, row quarter); item = (loop, 16-row k-step)
    {
      const int grp = warp >> 2, rq = warp & 3;
      const float al0 = S.alpha[2 * q], al1 = S.alpha[2 * q + 1];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        U.acc[mt][0] *= al0;
        U.acc[mt][1] *= al1;
        U.acc[mt][2] *= al0;
        U.acc[mt][3] *= al1;
      }
      int item = 0;
      for (int j = 0; j < depth; ++j) {
        const int nks = (M.loop[j].nrows + 15) >> 4;
        for (int ks = 0; ks < nks; ++ks, ++item) {
          if ((item & 3) != rq) continue;
          const uint8_t* base = &st.vc[j][(16 * ks) * kRowBytes + 4 * (8 * grp + g)];
          const uint32_t wa = *reinterpret_cast<const uint32_t*>(base + (q)*kRowBytes);
          const uint32_t wb = *reinterpret_cast<const uint32_t*>(base + (q + 4) * kRowBytes);
          const uint32_t wc = *reinterpret_cast<const uint32_t*>(base + (q + 8) * kRowBytes);
          const uint32_t wd = *reinterpret_cast<const uint32_t*>(base + (q + 12) * kRowBytes);
          const uint2 bp = *reinterpret_cast<const uint2*>(&S.pp[j][grp][ks][g][4 * q]);
          const uint32_t xab[2] = {__byte_perm(wa, wb, 0x5410), __byte_perm(wa, wb, 0x7632)};
          const uint32_t xcd[2] = {__byte_perm(wc, wd, 0x5410), __byte_perm(wc, wd, 0x7632)};
#pragma unroll
          for (int hbyte = 0; hbyte < 2; ++hbyte) {
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              const int mt = 2 * hbyte + sub;
              const uint32_t x1 = sub ? (xab[hbyte] >> 8) : xab[hbyte];
              const uint32_t x2 = sub ? (xcd[hbyte] >> 8) : xcd[hbyte];
              uint32_t A[4];
              A[0] = h2_sub1024(lop3_and_or(x1, 0x000F000Fu, 0x64006400u));
              A[1] = h2_hi_nibble(lop3_and_or(x1, 0x00F000F0u, 0x64006400u));
              A[2] = h2_sub1024(lop3_and_or(x2, 0x000F000Fu, 0x64006400u));
              A[3] = h2_hi_nibble(lop3_and_or(x2, 0x00F000F0u, 0x64006400u));
              mma16816(U.acc[mt], A, bp.x, bp.y);
            }
          }
        }
      }
    }
    // release the stage: every consumer warp is done reading it
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
  }
  if (cur_unit >= 0) finish_unit(a, S, U, Mprev, warp, lane);
}

__global__ void __launch_bounds__(kThreads, 1) attn_mma_kernel(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int C = a.n_ctas;
  const long long W = a.prefix[a.n_requests];
  const long long s0 = cta_start(blockIdx.x, W, C), e0 = cta_start(blockIdx.x + 1, W, C);
  if (s0 >= e0) return;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // P' rows of heads past the group size stay zero for the whole kernel
  for (int i = threadIdx.x; i < int(sizeof(S.pp) / 4); i += blockDim.x) reinterpret_cast<uint32_t*>(S.pp)[i] = 0u;
  __syncthreads();
  if (threadIdx.x >= kConsumers) {
    if (threadIdx.x == kConsumers) producer(a, S, s0, e0);
    return;
  }
  consumer(a, S, s0, e0);
}

}  // namespace mma_attn

cudaError_t launch_attn_mma(const AttnArgs& a, cudaStream_t stream) {
  using namespace mma_attn;
  const int smem = int(sizeof(Smem));
  static int configured = 0;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = 1;
  }
  attn_mma_kernel<<<a.n_ctas, kThreads, smem, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvq
