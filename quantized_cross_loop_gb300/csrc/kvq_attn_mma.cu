// kvq_attn_mma.cu — tensor-core decode attention over packed K/V.
//
// FlashLoop RFC (vllm-rlt issue #156) §3.2: historical K/V are read at the
// requested depth and reconstructed if compressed, scores scaled by
// 1/sqrt(head_dim); §3.3: readers consume the packed base/residual tiles
// directly during QK/PV instead of a BF16 shadow cache; §5: FP32 mass and
// accumulation. The dequantiser is the affine INT4 group code of §3.3
// (decode = min + scale * code).
//
// Design (ours). Each CTA holds two independent groups; a group is a virtual
// CTA of the flat (request, KV head, 64-token tile) work list of
// kvq_attn_common.cuh and owns a contiguous tile range.
//   producer warp   (one per group) one lane issues 1-D bulk TMA copies
//                   (cp.async.bulk with mbarrier transaction counts) of each
//                   tile's packed planes — per loop: K and V codes, K and V
//                   min/scale planes, and for a sparse loop its index slice —
//                   into the group's two stages.
//   4 consumer warps a warp owns 16 logical tokens of the tile through QK^T,
//                   softmax and PV; the dequantisation is folded into the
//                   contractions, since min and scale are constant along each:
//       S[t, h]  = sum_j [ sum_d c_j[t,d] * (q[h,d] * sK_j[d]) + sum_d q[h,d] * mK_j[d] ]
//       O[h, d]  = sum_j [ sum_t c_j[t,d] * (p[t,h] * sV_j[t]) + sum_t p[t,h] * mV_j[t] ]
//                   Codes enter mma.sync m16n8k16 (FP32 accumulate) as the FP16
//                   values 64 + c, made by OR-ing the nibble into the mantissa
//                   of 64.0; the offset is removed exactly: -64 * sum_d q*sK
//                   rides in the K-min MMA, -64 * sum_t p*sV is added in FP32.
//                   q (BF16) is exact in FP16; q*sK is carried exactly as the
//                   sum of two FP16 terms (hi = RN16(q*sK), lo = RN16(q*sK - hi)),
//                   so logits are exact up to FP32 accumulation. QK^T runs with
//                   tokens as M and the 8 query heads of a KV head as N; the
//                   softmax stays in the accumulator registers; p * sV becomes
//                   the PV B operand through movmatrix.trans; PV runs with
//                   channels as M. Both contractions run in token order: each
//                   thread addresses the stored row of its tokens (the rank of
//                   the token in the tile's 64-bit presence mask of a sparse
//                   loop), and a token without a row in a loop contributes
//                   neither logit nor value there.
// Each warp keeps its own online softmax (max, sum, PV accumulators) over its
// tokens; the group merges the four at the end of a unit. Per tile and group:
// one named barrier (K-min terms ready). Log2 domain, FP32 throughout.
//
// NVFP4 residual loops (INT4 codec PR review: E2M1 codes, an E4M3 scale per 16
// channels of a (row, head), an FP32 scale per stream), in the kNv
// instantiation. The scales vary along the contraction, so they scale the A
// operand instead of folding into Q or P:
//   QK^T: A = e2m1 * s_b (hardware E2M1 / E4M3 to FP16 conversions; the product
//         has at most six significant bits and lies in [2^-10, 2688], so it is
//         exact in FP16), B = q; the loop's logits are then scaled by s_t in FP32.
//   PV:   A = (e2m1 * 2^-14) * s_b, built from the nibble by bit placement
//         (FP16 bits (c & 7) << 9 | (c & 8) << 12 encode e2m1 * 2^-14 exactly,
//         and the product stays an exact FP16 multiple of 2^-24), B = RN16(p *
//         s_t * 2^14); NVFP4 has no zero point, so no min terms.
#include <cuda_fp16.h>

#include "kvq_attn_common.cuh"

namespace kvq {
namespace mma_attn {

constexpr int kLoops = 4;  // most loops staged per tile
constexpr int kGroups = 2;
constexpr int kGroupWarps = 4;
constexpr int kGroupThreads = kGroupWarps * 32;
constexpr int kStagesPerGroup = 2;
constexpr int kStages = kGroups * kStagesPerGroup;
constexpr int kConsumers = kGroups * kGroupThreads;
constexpr int kThreads = kConsumers + kGroups * 32;  // + one producer warp per group
constexpr int kMaxPairs = 2 * kLoops;                // (loop, K group) pairs of one tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitNs = 2000000000LL;  // bounded waits: 2 s, then flag and leave
constexpr uint32_t kMagic = 0x54005400u;     // FP16 64.0 in both halves

// Per-tile metadata written by the producer (int32 words).
//   [0] unit  [1] b  [2] h  [3] t0  [4] nvalid  [5] whole  [6] npairs
//   [7] first token of the tile read from the packed chain (later ones; earlier
//       tokens belong to the request's BF16 sink)
//   pair p (8 words from 8): loop index << 1 | group
//   loop j (8 words from 16 + 8j): nrows c0 g0 ngrp vrem irem sparse pbase
//       (c0: first stored row of the tile; under tile grouping of K, 64 x tile)
//   loop j formats (4 words from 16 + 8 kLoops + 4j): NVFP4 flags (1: K, 2: V),
//       K tensor scale, V tensor scale (float bits), byte offsets of the first
//       staged K | V block-scale row (low | high 16 bits)
constexpr int kMetaFmt = 16 + 8 * kLoops;
constexpr int kMetaWords = kMetaFmt + 4 * kLoops;

// One loop's staged planes of a tile (every field a multiple of 16 bytes, so
// that each starts on a 16-byte boundary for the bulk copies).
// An NVFP4 loop stages its E4M3 block scales (8 bytes per row, up to 528 bytes
// with the 16-byte rounding) over kmin..ksc (K) and vmin..vsc (V).
struct LoopStage {
  uint8_t kc[KVQ_TILE * kRowBytes];
  uint8_t vc[KVQ_TILE * kRowBytes];
  uint16_t kmin[2 * kD];
  uint16_t ksc[2 * kD];
  uint16_t vmin[144];  // 64 rows x 2 groups + 16 B rounding slack
  uint16_t vsc[144];
  int32_t idx[80];     // 64 indices + rounding slack
};
static_assert(sizeof(LoopStage) % 16 == 0, "loop stages keep 16-byte alignment");

struct __align__(128) Stage {
  LoopStage l[kLoops];
  int32_t meta[kMetaWords];
};

// Per warp and loop: first staged row of the warp's slice, row count, and the
// 16-bit presence mask of the slice's tokens (sparse loops).
struct SliceInfo {
  int32_t rb, cnt, bits, pad;
};

struct GroupSmem {
  __half q16[8][kD];                     // query of the current unit (BF16 values, exact in FP16)
  // sum_d q*mK - 64 sum_d q*sK per (pair, head), double-buffered by tile parity:
  // warp 0 writes the next tile's terms while other warps may still read these
  float kbias[2][kMaxPairs][8];
  float red[kGroupWarps][8];             // per-warp running max per head (unit-end merge)
  float lsum[kGroupWarps][8];
  float vbs[kGroupWarps][2][8];
  SliceInfo slice[kGroupWarps][kLoops];
  float fin[kGroupWarps][kD][8];         // end-of-unit sum of the warps' PV partials
};

struct Smem {
  Stage st[kStages];
  GroupSmem grp[kGroups];
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

// Named barrier of one consumer group (ids 1, 2).
__device__ __forceinline__ void group_sync(int grp) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kGroupThreads) : "memory");
}

// The group's barrier, returning whether any of its threads passed v = true.
__device__ __forceinline__ bool group_sync_or(int grp, bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred pi, po; setp.ne.u32 pi, %1, 0; bar.red.or.pred po, %2, %3, pi; selp.u32 %0, 1, 0, po; }"
      : "=r"(r)
      : "r"(uint32_t(v)), "r"(1 + grp), "n"(kGroupThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t m, uint32_t o) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(r) : "r"(a), "r"(m), "r"(o));
  return r;
}

// FP16 value 64 + (the nibble at bits 4..7 of each half of x).
__device__ __forceinline__ uint32_t nib(uint32_t x) { return lop3_and_or(x, 0x00F000F0u, kMagic); }

// Codes of a 32-bit word w (nibbles n0..n7, n0 = lowest channel) as FP16 pairs
// offset by 64: r[0] = {n0, n4}, r[1] = {n1, n5}, r[2] = {n2, n6}, r[3] = {n3, n7}.
__device__ __forceinline__ void unpack8(uint32_t w, uint32_t r[4]) {
  r[0] = nib(w << 4);
  r[1] = nib(w);
  r[2] = nib(w >> 4);
  r[3] = nib(w >> 8);
}

__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit values held one row pair per thread.
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ uint32_t h2u(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 u2h(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// Nibble c (0..3) of each 16-bit half of x as FP16 e2m1 * 2^-14: the nibble is
// moved to bits 12..15, then its magnitude bits to 9..11 under its sign at 15.
template <int C>
__device__ __forceinline__ uint32_t nv_pair(uint32_t x) {
  const uint32_t a = (C < 3 ? (x << (12 - 4 * C)) : x) & 0xF000F000u;
  return (a | (a >> 3)) & 0x8E008E00u;
}

// ---------------------------------------------------------------- producer
//
// One warp per group. Lane 8 j + c serves loop j with one 1-D bulk copy: c = 0
// the K code block, 1 the V code block, 2 the K min rows of the tile's groups
// (NVFP4 K: its E4M3 block scales, 8 B per row), 3 the K scale rows, 4 the V
// min rows (NVFP4 V: its block scales), 5 the V scale rows, 6 a sparse loop's
// index slice; row planes move in whole 16-byte units. All per-tile arithmetic
// comes before the wait for a free stage; after it the warp only issues the
// copies and writes the metadata, and lane 0 arrives (the copies issued one by
// one from a single thread after the wait kept the consumers waiting).

template <int DEPTH, bool kNv>
__device__ void producer(const AttnArgs& a, Smem& S, int grp, long long s0, long long e0, int lane) {
  const int j = lane >> 3, c = lane & 7;  // this lane's loop and copy
  int b = request_of(a.prefix, a.n_requests, s0);
  long long us = 0, ue = -1;  // current unit's tile range
  int h = 0, T = 0, unit = -1, nsink = 0;
  int nr = 0, kgr = 0;  // this lane's loop: stored rows; K groups per head (0: compact grouping)
  int rs = 0, gs = 0;   // plane strides: rows per head, K groups per head
  int fl = 0;           // NVFP4 flags (1: K, 2: V); the INT4 form never sees them (plan)
  float kst = 0.0f, vst = 0.0f;  // their tensor scales
  const int32_t* act = nullptr;
  const int32_t* dir = nullptr;
  const uint8_t *kc = nullptr, *vc = nullptr;
  const uint8_t *kmn = nullptr, *ksc = nullptr, *vmn = nullptr, *vsc = nullptr;
  long long it = 0;
  for (long long x = s0; x < e0; ++x, ++it) {
    if (x >= ue) {  // next unit: request b (skipping empty ones) and KV head h
      while (a.prefix[b + 1] <= x) ++b;
      const kvq_request& R = a.reqs[b];
      T = R.n_tokens;
      nsink = R.n_sink;
      const int nt = n_tiles_of(T);
      const long long rb = a.prefix[b];
      h = int((x - rb) / nt);
      us = rb + (long long)h * nt;
      ue = us + nt;
      unit = b * a.H + h;
      if (j < DEPTH) {
        const kvq_loop_ref& L = R.loop[j];
        nr = L.n_rows;
        kgr = (L.flags & KVQ_LOOP_K_TILE) ? k_groups_of(true, L.n_rows, T) : 0;
        rs = L.row_cap > 0 ? L.row_cap : L.n_rows;
        gs = L.kgroup_cap > 0 ? L.kgroup_cap : (kgr > 0 ? kgr : (L.n_rows + kG - 1) / kG);
        fl = kNv ? (((L.flags & KVQ_LOOP_K_NVFP4) ? 1 : 0) | ((L.flags & KVQ_LOOP_V_NVFP4) ? 2 : 0)) : 0;
        kst = (kNv && (fl & 1) && L.n_rows > 0 && c == 0) ? __ldg(reinterpret_cast<const float*>(L.k_scales)) : 0.0f;
        vst = (kNv && (fl & 2) && L.n_rows > 0 && c == 0) ? __ldg(reinterpret_cast<const float*>(L.v_scales)) : 0.0f;
        act = L.active_idx;
        dir = L.tile_dir;
        kc = L.k_codes;
        vc = L.v_codes;
        kmn = reinterpret_cast<const uint8_t*>(L.k_mins);
        ksc = reinterpret_cast<const uint8_t*>(L.k_scales);
        vmn = reinterpret_cast<const uint8_t*>(L.v_mins);
        vsc = reinterpret_cast<const uint8_t*>(L.v_scales);
      }
    }
    const int k = int(x - us);
    int c0 = 0, c1 = 0;
    bool bad = false;
    if (j < DEPTH) {
      if (act == nullptr) {
        c0 = k * KVQ_TILE;
        c1 = min(k * KVQ_TILE + KVQ_TILE, T);
      } else {
        c0 = __ldg(dir + k);
        c1 = __ldg(dir + k + 1);
      }
      if (c0 < 0 || c1 > nr || c0 > c1 || c1 - c0 > KVQ_TILE) {
        bad = true;
        c0 = c1 = 0;
      }
    }
    const int n = c1 - c0;
    // K groups of the tile's rows: under tile grouping the tile's own group k,
    // and word 1 is set so that a consumer's ((word1 + row) >> 6) - g0 is 0
    const bool kt = kgr > 0;
    const bool nk = kNv && (fl & 1), nv = kNv && (fl & 2);
    const int g0 = kt ? k : c0 / kG;
    const int ngrp = (j < DEPTH && n > 0 && !nk) ? (kt ? 1 : (c1 - 1) / kG - g0 + 1) : 0;  // INT4 K groups
    int pbase = 0, np = 0;  // pairs of the earlier loops, of all loops
#pragma unroll
    for (int jj = 0; jj < DEPTH; ++jj) {
      const int gj = __shfl_sync(0xffffffffu, ngrp, 8 * jj);
      pbase += jj < j ? gj : 0;
      np += gj;
    }
    const long long hr = (long long)h * rs + c0;  // first stored row of this head
    const long long koff = hr * 8, klo = koff & ~15LL;           // NVFP4 K block scales
    const long long voff = hr * (nv ? 8 : 4), vlo = voff & ~15LL;  // V rows (INT4 params or NVFP4 block scales)
    const long long ioff = (long long)c0 * 4, ilo = ioff & ~15LL;
    uint32_t bytes = 0;
    const uint8_t* src = nullptr;
    if (j < DEPTH && n > 0) {
      const long long gb = ((long long)h * gs + g0) * kD * 2;
      const uint32_t vbytes = uint32_t(((voff + (long long)n * (nv ? 8 : 4) + 15) & ~15LL) - vlo);
      switch (c) {
        case 0: bytes = uint32_t(n * kRowBytes); src = kc + hr * kRowBytes; break;
        case 1: bytes = uint32_t(n * kRowBytes); src = vc + hr * kRowBytes; break;
        case 2:
          if (nk) {
            bytes = uint32_t(((koff + (long long)n * 8 + 15) & ~15LL) - klo);
            src = kmn + klo;
          } else {
            bytes = uint32_t(ngrp * kD * 2);
            src = kmn + gb;
          }
          break;
        case 3:
          if (!nk) {
            bytes = uint32_t(ngrp * kD * 2);
            src = ksc + gb;
          }
          break;
        case 4: bytes = vbytes; src = vmn + vlo; break;
        case 5:
          if (!nv) {
            bytes = vbytes;
            src = vsc + vlo;
          }
          break;
        case 6:
          if (act != nullptr) {
            bytes = uint32_t(((ioff + (long long)n * 4 + 15) & ~15LL) - ilo);
            src = reinterpret_cast<const uint8_t*>(act) + ilo;
          }
          break;
        default: break;
      }
    }
    uint32_t total = bytes;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);

    const int s = grp * kStagesPerGroup + int(it & 1);
    const uint32_t ph = uint32_t((it >> 1) & 1);
    int ok = 1;
    if (lane == 0 && it >= kStagesPerGroup) ok = mbar_wait(&S.empty[s], ph ^ 1u) ? 1 : 0;
    if (!__shfl_sync(0xffffffffu, ok, 0)) {
      if (lane == 0) atomicOr(a.err, 8);
      return;
    }
    Stage& st = S.st[s];
    int32_t* M = st.meta;
    if (lane == 0) mbar_expect_tx(&S.full[s], total);
    __syncwarp();
    if (bytes > 0) {
      LoopStage& LS = st.l[j];
      void* dst = c == 0 ? (void*)LS.kc
                  : c == 1 ? (void*)LS.vc
                  : c == 2 ? (void*)LS.kmin
                  : c == 3 ? (void*)LS.ksc
                  : c == 4 ? (void*)LS.vmin
                  : c == 5 ? (void*)LS.vsc
                           : (void*)LS.idx;
      asm volatile(
          "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              smem_addr(dst)),
          "l"(src), "r"(bytes), "r"(smem_addr(&S.full[s]))
          : "memory");
    }
    // metadata
    if (lane == 0) {
      M[0] = unit;
      M[1] = b;
      M[2] = h;
      M[3] = k * KVQ_TILE;
      M[4] = min(KVQ_TILE, T - k * KVQ_TILE);
      M[5] = (us >= s0 && ue <= e0) ? 1 : 0;
      M[6] = np;
      M[7] = max(0, min(KVQ_TILE, nsink - k * KVQ_TILE));
    }
    if (j < DEPTH) {
      int32_t* LM = M + 16 + 8 * j;
      if (c == 0) {
        LM[0] = n;
        LM[1] = kt ? k * kG : c0;
        LM[2] = g0;
        LM[3] = ngrp;
        LM[4] = (n > 0 && !nv) ? int((voff - vlo) / 2) : 0;
        LM[5] = (n > 0 && act != nullptr) ? int((ioff - ilo) / 4) : 0;
        LM[6] = act != nullptr;
        LM[7] = pbase;
        if (kNv) {
          int32_t* LF = M + kMetaFmt + 4 * j;  // read by the NVFP4 form only
          LF[0] = fl;
          LF[1] = __float_as_int(kst);
          LF[2] = __float_as_int(vst);
          LF[3] = n > 0 ? (int(nk ? koff - klo : 0) | (int(nv ? voff - vlo : 0) << 16)) : 0;
        }
        if (bad) atomicOr(a.err, 4);
      } else if (c == 1 || c == 2) {
        if (c - 1 < ngrp) M[8 + pbase + c - 1] = (j << 1) | (c - 1);
      }
    }
    // the single expected arrival releases the metadata (ordered after every
    // lane's writes by the warp barrier); the phase completes once every copy
    // has delivered its bytes
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.full[s]);
  }
}

// ---------------------------------------------------------------- consumers

struct UnitState {
  float m[2];       // this warp's running max of heads 2q, 2q+1 (log2 units)
  float l[2];       // partial sums of exp2 of this thread's tokens for heads 2q, 2q+1
  float vb[2][2];   // partial V-min terms (with the -64 offset correction): [V group][head 2q / 2q+1]
  float acc[8][4];  // PV accumulators: 8 channel m-tiles x (2 rows x 2 heads)
};

struct UnitInfo {
  int unit, b, h, whole;
};

__device__ void load_unit_query(const AttnArgs& a, GroupSmem& G, int b, int h, int gt) {
  for (int i = gt; i < 8 * kD; i += kGroupThreads) {
    const int hh = i / kD, d = i % kD;
    float v = 0.0f;
    if (hh < a.g) v = bf16_bits_to_f32(a.q[((long long)b * a.Hq + (long long)h * a.g + hh) * kD + d]);
    G.q16[hh][d] = __float2half_rn(v);  // exact: a BF16 value in the FP16 range
  }
}

// Writes the unit's result: output rows (whole unit) or the group's partial slot.
// The four warps' online-softmax states are merged: each warp rescales its sums
// by exp2(m_warp - m_group) before they are added.
__device__ void finish_unit(const AttnArgs& a, GroupSmem& G, UnitState& U, const UnitInfo& M, int grp, int vcta,
                            int w, int lane) {
  const int gt = w * 32 + lane;
  const int g = lane >> 2, q = lane & 3;
  if (g == 0) {
    G.red[w][2 * q] = U.m[0];
    G.red[w][2 * q + 1] = U.m[1];
  }
  group_sync(grp);
  float mg[2], sc[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int hh = 2 * q + e;
    mg[e] = fmaxf(fmaxf(G.red[0][hh], G.red[1][hh]), fmaxf(G.red[2][hh], G.red[3][hh]));
    sc[e] = (mg[e] == -INFINITY || U.m[e] == -INFINITY) ? 0.f : exp2f(U.m[e] - mg[e]);
  }
  float l0 = U.l[0] * sc[0], l1 = U.l[1] * sc[1];
  float v00 = U.vb[0][0] * sc[0], v01 = U.vb[0][1] * sc[1], v10 = U.vb[1][0] * sc[0], v11 = U.vb[1][1] * sc[1];
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    v00 += __shfl_xor_sync(0xffffffffu, v00, off);
    v01 += __shfl_xor_sync(0xffffffffu, v01, off);
    v10 += __shfl_xor_sync(0xffffffffu, v10, off);
    v11 += __shfl_xor_sync(0xffffffffu, v11, off);
  }
  if (g == 0) {
    G.lsum[w][2 * q] = l0;
    G.lsum[w][2 * q + 1] = l1;
    G.vbs[w][0][2 * q] = v00;
    G.vbs[w][0][2 * q + 1] = v01;
    G.vbs[w][1][2 * q] = v10;
    G.vbs[w][1][2 * q + 1] = v11;
  }
#pragma unroll
  for (int vg = 0; vg < 2; ++vg)
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int ch = 64 * vg + 8 * g + 2 * mt;
      const float* c = U.acc[4 * vg + mt];
      *reinterpret_cast<float2*>(&G.fin[w][ch][2 * q]) = make_float2(c[0] * sc[0], c[1] * sc[1]);
      *reinterpret_cast<float2*>(&G.fin[w][ch + 1][2 * q]) = make_float2(c[2] * sc[0], c[3] * sc[1]);
    }
  group_sync(grp);
  const int gq = a.g;
  float* slot = a.partials + (size_t)(vcta + M.unit) * kSlotFloats;
  for (int i = gt; i < gq * kD; i += kGroupThreads) {
    const int hh = i / kD, d = i % kD, vg = d >> 6;
    const float lt = G.lsum[0][hh] + G.lsum[1][hh] + G.lsum[2][hh] + G.lsum[3][hh];
    const float vb = G.vbs[0][vg][hh] + G.vbs[1][vg][hh] + G.vbs[2][vg][hh] + G.vbs[3][vg][hh];
    const float o = (G.fin[0][d][hh] + G.fin[1][d][hh]) + (G.fin[2][d][hh] + G.fin[3][d][hh]) + vb;
    if (M.whole) {
      a.out[((long long)M.b * a.Hq + (long long)M.h * gq + hh) * kD + d] = o / lt;
      if (d == 0)
        a.stats[(long long)M.b * a.Hq + (long long)M.h * gq + hh] =
            make_float2(fmaxf(fmaxf(G.red[0][hh], G.red[1][hh]), fmaxf(G.red[2][hh], G.red[3][hh])), lt);
    } else {
      slot[2 * kMaxG + hh * kD + d] = o;
      if (d == 0) {
        slot[kMaxG + hh] = lt;
        slot[hh] = fmaxf(fmaxf(G.red[0][hh], G.red[1][hh]), fmaxf(G.red[2][hh], G.red[3][hh]));
      }
    }
  }
  group_sync(grp);
}

// Logits of the 16 staged rows (rb + g, rb + g + 8 per thread) of loop j against
// K group G: Q' = q * sK as exact FP16 hi + lo terms, codes unpacked from the
// two 16-byte chunks wa (row g) and wb (row g + 8); four accumulation chains.
__device__ __forceinline__ void qk_pass(const Stage& st, int j, int G, const uint32_t qp[16], const uint4 wa,
                                        const uint4 wb, int q, float e[4]) {
  const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w}, wB[4] = {wb.x, wb.y, wb.z, wb.w};
  float c[4][4] = {};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 sv4 = *reinterpret_cast<const uint4*>(&st.l[j].ksc[G * kD + 32 * q + 8 * i]);
    const uint32_t sp[4] = {__byte_perm(sv4.x, sv4.z, 0x5410), __byte_perm(sv4.x, sv4.z, 0x7632),
                            __byte_perm(sv4.y, sv4.w, 0x5410), __byte_perm(sv4.y, sv4.w, 0x7632)};
    uint32_t bh[4], bl[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 hv = __hmul2(u2h(qp[4 * i + k]), u2h(sp[k]));               // RN16(q * s)
      const __half2 lv = __hfma2(u2h(qp[4 * i + k]), u2h(sp[k]), __hneg2(hv));  // RN16(q * s - hi)
      bh[k] = h2u(hv);
      bl[k] = h2u(lv);
    }
    uint32_t ua[4], ub[4];
    unpack8(wA[i], ua);
    unpack8(wB[i], ub);
    const uint32_t A0[4] = {ua[0], ub[0], ua[1], ub[1]};
    const uint32_t A1[4] = {ua[2], ub[2], ua[3], ub[3]};
    mma16816(c[0], A0, bh[0], bh[1]);
    mma16816(c[1], A1, bh[2], bh[3]);
    mma16816(c[2], A0, bl[0], bl[1]);
    mma16816(c[3], A1, bl[2], bl[3]);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) e[k] = (c[0][k] + c[1][k]) + (c[2][k] + c[3][k]);
}

// Logits of rows ra (token g) and rc (token g + 8) of an NVFP4 K loop j: A =
// e2m1 * s_b (FP16, exact), B = q, two MMA chains; the sum is scaled by the
// stream's tensor scale st. krem: byte offset of the staged block-scale rows.
__device__ __forceinline__ void qk_pass_nv(const Stage& st, int j, const __half* qrow, int krem, int ra, int rc,
                                           const uint4 wa, const uint4 wb, int q, float tscale, float e[4]) {
  const uint8_t* ks = reinterpret_cast<const uint8_t*>(st.l[j].kmin) + krem;  // row r: 8 bytes at 8 r
  // blocks 2q and 2q + 1 of each row: channels 32q .. 32q + 31, this thread's
  const uint32_t sa2 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(ks + 8 * ra + 2 * q));
  const uint32_t sc2 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(ks + 8 * rc + 2 * q));
  const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w}, wB[4] = {wb.x, wb.y, wb.z, wb.w};
  float c[2][4] = {};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 sa = i < 2 ? __low2half2(u2h(sa2)) : __high2half2(u2h(sa2));
    const __half2 sc = i < 2 ? __low2half2(u2h(sc2)) : __high2half2(u2h(sc2));
    uint32_t ua[4], ub[4];  // channel pairs (2k, 2k + 1) of word i, scaled
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ua[k] = h2u(__hmul2(u2h(e2m1x2_to_f16x2(wA[i] >> (8 * k))), sa));
      ub[k] = h2u(__hmul2(u2h(e2m1x2_to_f16x2(wB[i] >> (8 * k))), sc));
    }
    const uint4 qv = *reinterpret_cast<const uint4*>(qrow + 32 * q + 8 * i);  // q of channels 32q + 8i .. + 7
    const uint32_t A0[4] = {ua[0], ub[0], ua[1], ub[1]};
    const uint32_t A1[4] = {ua[2], ub[2], ua[3], ub[3]};
    mma16816(c[0], A0, qv.x, qv.y);
    mma16816(c[1], A1, qv.z, qv.w);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) e[k] = (c[0][k] + c[1][k]) * tscale;
}

template <int DEPTH, bool kNv, bool kSp>
__device__ void consumer(const AttnArgs& a, Smem& S, int grp, int vcta, long long s0, long long e0) {
  const int gt = threadIdx.x - grp * kGroupThreads;  // thread within the group
  const int w = gt >> 5, lane = gt & 31;
  const int g = lane >> 2, q = lane & 3;
  const int gq = a.g;
  const float lsc = a.scale * kLog2e;
  GroupSmem& Gs = S.grp[grp];
  UnitState U;
  int cur_unit = -1;
  UnitInfo Mprev = {-1, 0, 0, 0};
  uint32_t qp[16];  // q of head g, channels 32q..32q+31, as FP16 pairs in fragment order
  long long it = 0;

  for (long long x = s0; x < e0; ++x, ++it) {
    const int s = grp * kStagesPerGroup + int(it & 1);
    const uint32_t ph = uint32_t((it >> 1) & 1);
    // a wait that ran out ends the whole group together (its warps meet at the group's barriers)
    if (group_sync_or(grp, !mbar_wait(&S.full[s], ph))) {
      if (gt == 0) atomicOr(a.err, 8);
      return;
    }
    const Stage& st = S.st[s];
    const int4 m0 = *reinterpret_cast<const int4*>(&st.meta[0]);
    const int4 m1 = *reinterpret_cast<const int4*>(&st.meta[4]);
    const int unit = m0.x, t0 = m0.w, nvalid = m1.x, npairs = m1.z, tfirst = m1.w;
    if (unit != cur_unit) {
      if (cur_unit >= 0) finish_unit(a, Gs, U, Mprev, grp, vcta, w, lane);
      cur_unit = unit;
      Mprev.unit = unit;
      Mprev.b = m0.y;
      Mprev.h = m0.z;
      Mprev.whole = m1.y;
      U.m[0] = U.m[1] = -INFINITY;
      U.l[0] = U.l[1] = 0.f;
      U.vb[0][0] = U.vb[0][1] = U.vb[1][0] = U.vb[1][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) U.acc[mt][e] = 0.f;
      load_unit_query(a, Gs, Mprev.b, Mprev.h, gt);
      group_sync(grp);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half* qr = &Gs.q16[g][32 * q + 8 * i];
        qp[4 * i + 0] = h2u(__halves2half2(qr[0], qr[4]));
        qp[4 * i + 1] = h2u(__halves2half2(qr[1], qr[5]));
        qp[4 * i + 2] = h2u(__halves2half2(qr[2], qr[6]));
        qp[4 * i + 3] = h2u(__halves2half2(qr[3], qr[7]));
      }
    }

    // ---- K-min terms of every (loop, group) pair, by warp 0 of the group, in one
    // MMA chain: rows 0..7 = the pairs' mins, rows 8..15 = their scales times
    // -64 (removing the code offset); K = channels, N = heads.
    if (w == 0) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      const bool live = g < npairs;
      const int pj = live ? st.meta[8 + g] : 0;
      const uint16_t* mrow = &st.l[pj >> 1].kmin[(pj & 1) * kD];
      const uint16_t* srow = &st.l[pj >> 1].ksc[(pj & 1) * kD];
      const __half2 m64 = __float2half2_rn(-64.f);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t av[4] = {0u, 0u, 0u, 0u};
        if (live) {
          av[0] = *reinterpret_cast<const uint32_t*>(mrow + 16 * kk + 2 * q);
          av[1] = h2u(__hmul2(u2h(*reinterpret_cast<const uint32_t*>(srow + 16 * kk + 2 * q)), m64));
          av[2] = *reinterpret_cast<const uint32_t*>(mrow + 16 * kk + 2 * q + 8);
          av[3] = h2u(__hmul2(u2h(*reinterpret_cast<const uint32_t*>(srow + 16 * kk + 2 * q + 8)), m64));
        }
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&Gs.q16[g][16 * kk + 2 * q]);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&Gs.q16[g][16 * kk + 2 * q + 8]);
        mma16816(c, av, b0, b1);
      }
      if (live) *reinterpret_cast<float2*>(&Gs.kbias[it & 1][g][2 * q]) = make_float2(c[0] + c[2], c[1] + c[3]);
    }

    // ---- QK^T of the warp's 16 tokens [16w, 16w + 16) over every loop
    // logits in the accumulator layout: sv[0] (token g, head 2q), sv[1] (g, 2q+1),
    // sv[2] (g + 8, 2q), sv[3] (g + 8, 2q + 1)
    float sv[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t pinfo = 0;  // per loop 4 bits: tokens g / g+8 present, and their K group
    for (int j = 0; j < DEPTH; ++j) {
      const int4 la = *reinterpret_cast<const int4*>(&st.meta[16 + 8 * j]);
      const int4 lb = *reinterpret_cast<const int4*>(&st.meta[20 + 8 * j]);
      const int c0 = la.y, g0 = la.z, ngrp = la.w, irem = lb.y, sparse = lb.z;
      int rb, cnt, bits;
      if (!sparse) {
        rb = 16 * w;
        cnt = max(0, min(16, nvalid - 16 * w));
        bits = cnt >= 16 ? 0xFFFF : ((1 << cnt) - 1);
      } else {
        // presence of the tile's tokens in this loop, from its staged index slice
        // (at most 64 entries: two per lane, OR-reduced over the warp)
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int i0 = 0; i0 < KVQ_TILE; i0 += 32) {
          const int i = i0 + lane;
          const int u = i < la.x ? st.l[j].idx[irem + i] - t0 : -1;
          if (u >= 0 && u < 32) lo |= 1u << u;
          if (u >= 32 && u < KVQ_TILE) hi |= 1u << (u - 32);
        }
        lo = __reduce_or_sync(0xffffffffu, lo);
        hi = __reduce_or_sync(0xffffffffu, hi);
        const unsigned long long mk = (unsigned long long)hi << 32 | lo;
        bits = int((mk >> (16 * w)) & 0xFFFFull);
        rb = __popcll(mk & ((1ull << (16 * w)) - 1ull));
        cnt = __popc(bits);
      }
      if (lane == 0) Gs.slice[w][j] = SliceInfo{rb, cnt, bits, 0};
      if (cnt == 0) continue;
      float e[4];
      if (kNv && (st.meta[kMetaFmt + 4 * j] & 1)) {  // NVFP4 K: no groups, no min terms
        const int ra = rb + min(__popc(bits & ((1 << g) - 1)), cnt - 1);
        const int rc = rb + min(__popc(bits & ((1 << (g + 8)) - 1)), cnt - 1);
        const uint4 wa = *reinterpret_cast<const uint4*>(&st.l[j].kc[ra * kRowBytes + 16 * q]);
        const uint4 wb = *reinterpret_cast<const uint4*>(&st.l[j].kc[rc * kRowBytes + 16 * q]);
        const int4 lf = *reinterpret_cast<const int4*>(&st.meta[kMetaFmt + 4 * j]);
        qk_pass_nv(st, j, &Gs.q16[g][0], lf.w & 0xFFFF, ra, rc, wa, wb, q, __int_as_float(lf.y), e);
        if ((bits >> g) & 1) {
          sv[0] += e[0];
          sv[1] += e[1];
        }
        if ((bits >> (g + 8)) & 1) {
          sv[2] += e[2];
          sv[3] += e[3];
        }
        continue;
      }
      // K groups of the slice's rows, relative to the tile's first group
      const int ga = ((c0 + rb) >> 6) - g0;
      const int gb = ((c0 + rb + cnt - 1) >> 6) - g0;
      const bool split = gb != ga;
      // A: the stored rows of the warp's tokens g and g + 8 (a sparse loop's r-th
      // present token sits in row rb + r; an absent token reads a valid row whose
      // logit is then dropped), the 16 bytes of chunk q
      const int ra = rb + min(__popc(bits & ((1 << g) - 1)), cnt - 1);
      const int rc = rb + min(__popc(bits & ((1 << (g + 8)) - 1)), cnt - 1);
      const uint4 wa = *reinterpret_cast<const uint4*>(&st.l[j].kc[ra * kRowBytes + 16 * q]);
      const uint4 wb = *reinterpret_cast<const uint4*>(&st.l[j].kc[rc * kRowBytes + 16 * q]);
      qk_pass(st, j, ga, qp, wa, wb, q, e);
      const int Ga = ((c0 + ra) >> 6) - g0, Gc = ((c0 + rc) >> 6) - g0;
      if (split) {  // rows of the second K group: a second pass with that group's Q'
        float f[4];
        qk_pass(st, j, gb, qp, wa, wb, q, f);
        if (Ga != ga) e[0] = f[0], e[1] = f[1];
        if (Gc != ga) e[2] = f[2], e[3] = f[3];
      }
      uint32_t pi = 0;
      if ((bits >> g) & 1) {
        sv[0] += e[0];
        sv[1] += e[1];
        pi |= 1u | (uint32_t(Ga) << 1);
      }
      if ((bits >> (g + 8)) & 1) {
        sv[2] += e[2];
        sv[3] += e[3];
        pi |= (1u | (uint32_t(Gc) << 1)) << 2;
      }
      (void)ngrp;
      pinfo |= pi << (4 * j);
    }
    group_sync(grp);  // K-min terms and slice info visible

    // ---- logits in log2 units and this warp's max per head
    float mt0, mt1;
    {
#pragma unroll
      for (int j = 0; j < DEPTH; ++j) {
        const int pbase = st.meta[16 + 8 * j + 7];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t f = (pinfo >> (4 * j + 2 * half)) & 3u;
          if (f & 1u) {
            const float2 kb = *reinterpret_cast<const float2*>(&Gs.kbias[it & 1][pbase + int(f >> 1)][2 * q]);
            sv[2 * half] += kb.x;
            sv[2 * half + 1] += kb.y;
          }
        }
      }
      const bool h0ok = 2 * q < gq, h1ok = 2 * q + 1 < gq;
      const bool t0ok = 16 * w + g < nvalid && 16 * w + g >= tfirst;
      const bool t1ok = 16 * w + g + 8 < nvalid && 16 * w + g + 8 >= tfirst;
      sv[0] = (t0ok && h0ok) ? sv[0] * lsc : -INFINITY;
      sv[1] = (t0ok && h1ok) ? sv[1] * lsc : -INFINITY;
      sv[2] = (t1ok && h0ok) ? sv[2] * lsc : -INFINITY;
      sv[3] = (t1ok && h1ok) ? sv[3] * lsc : -INFINITY;
      if (kSp && a.sel_mask != nullptr) {  // sparse decode: only the query head's selected keys
        const int tb = t0 + 16 * w;   // the warp's first token: its 16 tokens share one mask word
        // a request longer than the masks cover (the sparse path refuses it) selects nothing here
        const bool in = (tb >> 5) < a.mask_words;
        const uint32_t* mw = a.sel_mask + ((long long)Mprev.b * a.Hq + (long long)Mprev.h * gq) * a.mask_words + (tb >> 5);
        const uint32_t w0 = (in && h0ok) ? __ldg(mw + (long long)(2 * q) * a.mask_words) >> (tb & 31) : 0u;
        const uint32_t w1 = (in && h1ok) ? __ldg(mw + (long long)(2 * q + 1) * a.mask_words) >> (tb & 31) : 0u;
        if (!((w0 >> g) & 1u)) sv[0] = -INFINITY;
        if (!((w1 >> g) & 1u)) sv[1] = -INFINITY;
        if (!((w0 >> (g + 8)) & 1u)) sv[2] = -INFINITY;
        if (!((w1 >> (g + 8)) & 1u)) sv[3] = -INFINITY;
      }
      if (kSp && a.logits != nullptr) {  // sparse decode reference pass: every logit, for the selection
        const int ta = t0 + 16 * w + g, tc = ta + 8;
        float* lr = a.logits + ((long long)Mprev.b * a.Hq + (long long)Mprev.h * gq) * a.logit_stride;
        if (t0ok && h0ok && ta < a.logit_stride) lr[(long long)(2 * q) * a.logit_stride + ta] = sv[0];
        if (t0ok && h1ok && ta < a.logit_stride) lr[(long long)(2 * q + 1) * a.logit_stride + ta] = sv[1];
        if (t1ok && h0ok && tc < a.logit_stride) lr[(long long)(2 * q) * a.logit_stride + tc] = sv[2];
        if (t1ok && h1ok && tc < a.logit_stride) lr[(long long)(2 * q + 1) * a.logit_stride + tc] = sv[3];
      }
      mt0 = fmaxf(sv[0], sv[2]);
      mt1 = fmaxf(sv[1], sv[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {  // this warp's 16 tokens
        mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, off));
        mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, off));
      }
    }

    // ---- online softmax of the warp in registers, then PV over every loop
    {
      const float mn0 = fmaxf(U.m[0], mt0), mn1 = fmaxf(U.m[1], mt1);
      const float al0 = (U.m[0] == -INFINITY) ? 0.f : exp2f(U.m[0] - mn0);
      const float al1 = (U.m[1] == -INFINITY) ? 0.f : exp2f(U.m[1] - mn1);
      U.m[0] = mn0;
      U.m[1] = mn1;
      float p[4];
      p[0] = sv[0] == -INFINITY ? 0.f : exp2f(sv[0] - mn0);
      p[1] = sv[1] == -INFINITY ? 0.f : exp2f(sv[1] - mn1);
      p[2] = sv[2] == -INFINITY ? 0.f : exp2f(sv[2] - mn0);
      p[3] = sv[3] == -INFINITY ? 0.f : exp2f(sv[3] - mn1);
      U.l[0] = U.l[0] * al0 + (p[0] + p[2]);
      U.l[1] = U.l[1] * al1 + (p[1] + p[3]);
#pragma unroll
      for (int vg = 0; vg < 2; ++vg) {
        U.vb[vg][0] *= al0;
        U.vb[vg][1] *= al1;
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        U.acc[mt][0] *= al0;
        U.acc[mt][1] *= al1;
        U.acc[mt][2] *= al0;
        U.acc[mt][3] *= al1;
      }
      for (int j = 0; j < DEPTH; ++j) {
        const SliceInfo si = Gs.slice[w][j];
        if (si.cnt == 0) continue;
        const int vrem = st.meta[16 + 8 * j + 4];
        const int bits = si.bits, rb = si.rb, cnt = si.cnt;
        if (kNv && (st.meta[kMetaFmt + 4 * j] & 2)) {  // NVFP4 V
          // stored rows of the tokens 2q, 2q+1, 2q+8, 2q+9 (an absent token reads a
          // valid row against a zero P')
          const int r0 = rb + min(__popc(bits & ((1 << (2 * q)) - 1)), cnt - 1);
          const int r1 = rb + min(__popc(bits & ((2 << (2 * q)) - 1)), cnt - 1);
          const int r2 = rb + min(__popc(bits & ((1 << (2 * q + 8)) - 1)), cnt - 1);
          const int r3 = rb + min(__popc(bits & ((2 << (2 * q + 8)) - 1)), cnt - 1);
          const int4 lf = *reinterpret_cast<const int4*>(&st.meta[kMetaFmt + 4 * j]);
          const float st14 = __int_as_float(lf.z) * 16384.0f;  // s_t * 2^14 (the codes carry 2^-14)
          const uint8_t* vs = reinterpret_cast<const uint8_t*>(st.l[j].vmin) + (lf.w >> 16);
          uint32_t rr[2];  // [token half] = {P'(token, 2q), P'(token, 2q+1)}
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const bool ok = (bits >> (g + 8 * half)) & 1;
            rr[half] = h2u(__floats2half2_rn(ok ? p[2 * half] * st14 : 0.f, ok ? p[2 * half + 1] * st14 : 0.f));
          }
          const uint32_t B0 = transpose8x8(rr[0]), B1 = transpose8x8(rr[1]);
          const uint8_t* base = &st.l[j].vc[0];
#pragma unroll
          for (int vg = 0; vg < 2; ++vg) {
            const int blk = 4 * vg + (g >> 1);  // the 16-channel block of channels 64 vg + 8 g .. + 7
            const __half2 S01 = u2h(e4m3x2_to_f16x2(uint32_t(vs[8 * r0 + blk]) | (uint32_t(vs[8 * r1 + blk]) << 8)));
            const __half2 S89 = u2h(e4m3x2_to_f16x2(uint32_t(vs[8 * r2 + blk]) | (uint32_t(vs[8 * r3 + blk]) << 8)));
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(base + r0 * kRowBytes + 4 * (8 * vg + g));
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(base + r1 * kRowBytes + 4 * (8 * vg + g));
            const uint32_t w2 = *reinterpret_cast<const uint32_t*>(base + r2 * kRowBytes + 4 * (8 * vg + g));
            const uint32_t w3 = *reinterpret_cast<const uint32_t*>(base + r3 * kRowBytes + 4 * (8 * vg + g));
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              const uint32_t x = __byte_perm(w0, w1, hb ? 0x7632 : 0x5410);
              const uint32_t y = __byte_perm(w2, w3, hb ? 0x7632 : 0x5410);
              const uint32_t A0[4] = {h2u(__hmul2(u2h(nv_pair<0>(x)), S01)), h2u(__hmul2(u2h(nv_pair<1>(x)), S01)),
                                      h2u(__hmul2(u2h(nv_pair<0>(y)), S89)), h2u(__hmul2(u2h(nv_pair<1>(y)), S89))};
              const uint32_t A1[4] = {h2u(__hmul2(u2h(nv_pair<2>(x)), S01)), h2u(__hmul2(u2h(nv_pair<3>(x)), S01)),
                                      h2u(__hmul2(u2h(nv_pair<2>(y)), S89)), h2u(__hmul2(u2h(nv_pair<3>(y)), S89))};
              mma16816(U.acc[4 * vg + 2 * hb], A0, B0, B1);
              mma16816(U.acc[4 * vg + 2 * hb + 1], A1, B0, B1);
            }
          }
          continue;
        }
        // P' = p * sV per V group for the warp's tokens g and g + 8 (zero for a token
        // with no row in this loop), and the V-min terms
        uint32_t r[2][2];  // [V group][token half] = {P'(token, 2q), P'(token, 2q+1)}
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int tok = g + 8 * half;
          const bool ok = (bits >> tok) & 1;
          const int vi = vrem + 2 * (rb + min(__popc(bits & ((1 << tok) - 1)), cnt - 1));
          const uint32_t sraw = ok ? *reinterpret_cast<const uint32_t*>(&st.l[j].vsc[vi]) : 0u;
          const uint32_t mraw = ok ? *reinterpret_cast<const uint32_t*>(&st.l[j].vmin[vi]) : 0u;
          const float p0 = ok ? p[2 * half] : 0.f, p1 = ok ? p[2 * half + 1] : 0.f;
          const __half2 pp = __floats2half2_rn(p0, p1);
          const __half2 sv2 = u2h(sraw);
          const float2 mv = __half22float2(u2h(mraw));
#pragma unroll
          for (int vg = 0; vg < 2; ++vg) {
            const __half2 sg = vg == 0 ? __low2half2(sv2) : __high2half2(sv2);
            const __half2 pv = __hmul2(pp, sg);
            r[vg][half] = h2u(pv);
            const float2 pf = __half22float2(pv);
            const float mg = vg == 0 ? mv.x : mv.y;
            U.vb[vg][0] = fmaf(p0, mg, fmaf(-64.f, pf.x, U.vb[vg][0]));
            U.vb[vg][1] = fmaf(p1, mg, fmaf(-64.f, pf.y, U.vb[vg][1]));
          }
        }
        // B operands (k = tokens, n = heads) by 8x8 transposes of the (token, head) blocks
        const uint32_t B00 = transpose8x8(r[0][0]), B01 = transpose8x8(r[0][1]);
        const uint32_t B10 = transpose8x8(r[1][0]), B11 = transpose8x8(r[1][1]);
        // A: V codes of the stored rows of tokens 2q, 2q+1, 2q+8, 2q+9 (an absent
        // token reads a valid row against a zero P'); thread g takes word 8*vg + g of
        // each row (channels 64vg + 8g .. +7)
        const uint8_t* base = &st.l[j].vc[0];
        const int o0 = (rb + min(__popc(bits & ((1 << (2 * q)) - 1)), cnt - 1)) * kRowBytes;
        const int o1 = (rb + min(__popc(bits & ((2 << (2 * q)) - 1)), cnt - 1)) * kRowBytes;
        const int o2 = (rb + min(__popc(bits & ((1 << (2 * q + 8)) - 1)), cnt - 1)) * kRowBytes;
        const int o3 = (rb + min(__popc(bits & ((2 << (2 * q + 8)) - 1)), cnt - 1)) * kRowBytes;
        uint32_t wv[2][4];
#pragma unroll
        for (int vg = 0; vg < 2; ++vg) {
          wv[vg][0] = *reinterpret_cast<const uint32_t*>(base + o0 + 4 * (8 * vg + g));
          wv[vg][1] = *reinterpret_cast<const uint32_t*>(base + o1 + 4 * (8 * vg + g));
          wv[vg][2] = *reinterpret_cast<const uint32_t*>(base + o2 + 4 * (8 * vg + g));
          wv[vg][3] = *reinterpret_cast<const uint32_t*>(base + o3 + 4 * (8 * vg + g));
        }
#pragma unroll
        for (int vg = 0; vg < 2; ++vg) {
          const uint32_t b0 = vg == 0 ? B00 : B10, b1 = vg == 0 ? B01 : B11;
          const uint32_t x[2] = {__byte_perm(wv[vg][0], wv[vg][1], 0x5410), __byte_perm(wv[vg][0], wv[vg][1], 0x7632)};
          const uint32_t y[2] = {__byte_perm(wv[vg][2], wv[vg][3], 0x5410), __byte_perm(wv[vg][2], wv[vg][3], 0x7632)};
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const uint32_t A0[4] = {nib(x[hb] << 4), nib(x[hb]), nib(y[hb] << 4), nib(y[hb])};
            const uint32_t A1[4] = {nib(x[hb] >> 4), nib(x[hb] >> 8), nib(y[hb] >> 4), nib(y[hb] >> 8)};
            mma16816(U.acc[4 * vg + 2 * hb], A0, b0, b1);
            mma16816(U.acc[4 * vg + 2 * hb + 1], A1, b0, b1);
          }
        }
      }
    }
    // release the stage: every warp of the group is done reading it
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
  }
  if (cur_unit >= 0) finish_unit(a, Gs, U, Mprev, grp, vcta, w, lane);
}

// kSp: the instantiation that reads the sparse-decode key masks and writes the
// reference pass's logits (the dense calls run the one without those branches)
template <int DEPTH, bool kNv, bool kSp>
__global__ void __launch_bounds__(kThreads, 1) attn_mma_kernel(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  if (a.dispatch == 2 && !(*a.flags & 2)) return;  // no NVFP4 loop in the call: the INT4 kernel ran
  const int C = a.n_ctas;  // virtual CTAs: two per block
  const long long W = a.prefix[a.n_requests];
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kGroupWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  int grp;
  bool producer_warp;
  if (threadIdx.x < kConsumers) {
    grp = threadIdx.x / kGroupThreads;
    producer_warp = false;
  } else {
    grp = (threadIdx.x - kConsumers) >> 5;
    producer_warp = true;
  }
  const int vcta = kGroups * blockIdx.x + grp;
  const long long s0 = cta_start(vcta, W, C), e0 = cta_start(vcta + 1, W, C);
  if (s0 >= e0) return;
  if (producer_warp) {
    producer<DEPTH, kNv>(a, S, grp, s0, e0, threadIdx.x & 31);
    return;
  }
  consumer<DEPTH, kNv, kSp>(a, S, grp, vcta, s0, e0);
}

template <int DEPTH, bool kNv, bool kSp>
cudaError_t launch_depth(const AttnArgs& a, cudaStream_t stream) {
  const int smem = int(sizeof(Smem));
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_mma_kernel<DEPTH, kNv, kSp>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  attn_mma_kernel<DEPTH, kNv, kSp><<<a.n_ctas / kGroups, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

// the NVFP4-reading instantiation only when the caller says the table may
// hold NVFP4 loops (the INT4 one refuses them: error bit 64, NaN output)
template <bool kSp>
cudaError_t launch_form(const AttnArgs& a, cudaStream_t stream) {
  switch (a.depth * 2 + (a.nvfp4 ? 1 : 0)) {
    case 2: return launch_depth<1, false, kSp>(a, stream);
    case 3: return launch_depth<1, true, kSp>(a, stream);
    case 4: return launch_depth<2, false, kSp>(a, stream);
    case 5: return launch_depth<2, true, kSp>(a, stream);
    case 6: return launch_depth<3, false, kSp>(a, stream);
    case 7: return launch_depth<3, true, kSp>(a, stream);
    case 8: return launch_depth<4, false, kSp>(a, stream);
    case 9: return launch_depth<4, true, kSp>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mma_attn

int mma_virtual_ctas_per_block() { return mma_attn::kGroups; }

cudaError_t launch_attn_mma(const AttnArgs& a, cudaStream_t stream) {
  using namespace mma_attn;
  if (!a.general && !a.nvfp4) {
    if (a.tcgen05 && a.sel_mask == nullptr && a.logits == nullptr) return launch_attn_tcgen05(a, stream);
    return launch_attn_tc(a, stream);
  }
  const cudaError_t e = (a.sel_mask != nullptr || a.logits != nullptr) ? launch_form<true>(a, stream)
                                                                        : launch_form<false>(a, stream);
  if (e == cudaErrorInvalidValue) return e;
  count_launch();
  return e;
}

}  // namespace kvq
