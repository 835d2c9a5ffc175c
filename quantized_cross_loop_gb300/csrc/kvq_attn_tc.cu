// kvq_attn_tc.cu — tensor-core decode attention over packed INT4 K/V chains,
// with the dequantisation folded into the contractions and the codes fed to
// the tensor cores as FP16 subnormals.
//
// FlashLoop RFC (vllm-rlt issue #156) §3.2: historical K/V are read at the
// requested depth and reconstructed if compressed, scores scaled by
// 1/sqrt(head_dim); §3.3: readers consume the packed base/residual tiles
// directly during QK/PV, and the dequantiser is the affine INT4 group code
// decode = min + scale * code; §5: FP32 mass and accumulation.
//
// Work list, partial slots, plan and merge are those of kvq_attn_common.cuh.
// A CTA holds two independent groups (virtual CTAs); a group is two producer
// warps, which stage alternate 64-token tiles' packed planes (codes, min and
// scale planes, sparse index slices) into the group's two-stage ring with 1-D
// bulk copies, and four consumer warps, each owning 16 tokens of the tile.
//
// Codes as subnormals. The nibble of channel c sits at bits 0..3 of its byte
// when c is even and at bits 4..7 when c is odd. AND-ing a 32-bit word of
// codes with 0x000F000F (or 0x00F000F0) leaves in each 16-bit half a nibble
// whose FP16 value is n * 2^-24 (or n * 2^-20): an exact subnormal, with no
// offset to remove. One shift and four ANDs give eight codes. (The tensor
// cores keep FP16 subnormal inputs exactly.)
//
// QK^T (per loop j, K group G of the tile's stored rows; tokens as M, columns
// as N, channels as K):
//   S[t, h] = sum_j [ sum_d c_j[t, d] * (q[h, d] * sK_j[d]) + sum_d q[h, d] * mK_j[d] ]
//   B = q * sK as an exact FP16 pair hi + lo (hi = RN16(q s), lo = RN16(q s - hi)),
//   divided by 16 for the odd channels (their codes carry 2^-20), so every
//   product is n * q * s * 2^-24; for up to four query heads the columns are
//   (head, hi | lo) pairs, and eight heads take two column blocks. The K-min term
//   q . mK is one more k-step: A = 2^-14 at k = 0 for a token stored in the
//   loop, B = (q . mK) * 2^-10 split into FP16 hi + lo. The B fragments and the
//   K-min terms are built once per tile by the group (not per warp); a token
//   without a row in a sparse loop gets an all-zero A row. The logits
//   accumulate over the loops in the MMA accumulators (scale 2^-24).
// Softmax: per warp, FP32, log2 domain, in the accumulator layout (a thread
//   holds tokens g, g + 8 and one query head, or two with eight heads); the four
//   warps' states are merged at the end of a unit.
// PV (per loop; channels as M, tokens as K, (query head, V group) as N):
//   O[d, h] = sum_j [ sum_t c_j[t, d] * (p[t, h] * sV_j[t, vg(d)]) + sum_t p[t, h] * mV_j[t, vg(d)] ]
//   B = P' = RN16(p * sV) through movmatrix transposes, A = the V codes of four
//   tokens paired by byte permutes; even channels come out scaled by 2^-24,
//   odd ones by 2^-20, undone at the end. The V-min terms are FP32 FMAs.
#include <cuda_fp16.h>

#include "kvq_attn_common.cuh"

namespace kvq {
namespace tc_attn {

constexpr int kLoops = 4;  // most loops staged per tile
constexpr int kGroups = 2;
constexpr int kGroupWarps = 4;
constexpr int kGroupThreads = kGroupWarps * 32;
constexpr int kStagesPerGroup = 2;
constexpr int kStages = kGroups * kStagesPerGroup;
constexpr int kConsumers = kGroups * kGroupThreads;
constexpr int kProducers = 2;                         // producer warps per group: one per stage
constexpr int kThreads = kConsumers + kGroups * kProducers * 32;
constexpr int kMaxPairs = 1 + 2 * (kLoops - 1);      // (loop, K group) pairs of a tile: loop 1 is dense
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitNs = 2000000000LL;  // bounded waits: 2 s, then flag and leave
constexpr uint32_t kLoMask = 0x000F000Fu;    // even channels: FP16 n * 2^-24
constexpr uint32_t kHiMask = 0x00F000F0u;    // odd channels:  FP16 n * 2^-20
constexpr uint32_t kKbA = 0x0400u;           // FP16 2^-14: the A entry of the K-min k-step

// Per-tile metadata written by the producer (int32 words).
//   [0] unit  [1] b  [2] h  [3] t0  [4] nvalid  [5] whole  [6] npairs
//   [7] first token of the tile read from the packed chain (earlier tokens
//       belong to the request's BF16 sink)
//   pair p (7 words from 8): loop index << 1 | group
//   loop j (8 words from 16 + 8j): nrows c0 g0 ngrp vrem irem sparse pbase
//       (c0: first stored row of the tile; under tile grouping of K, 64 x tile)
constexpr int kMetaWords = 16 + 8 * kLoops;

// One loop's staged planes of a tile (every field a multiple of 16 bytes).
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

struct __align__(16) GroupSmem {
  union {
    // B fragments of QK^T: [pair][head block][word i][lane] = {k-step (i, 0): b0, b1; (i, 1): b0, b1}
    uint4 qf[kMaxPairs][2][4][32];
    float fin[kGroupWarps][kD][8];  // end-of-unit sum of the warps' PV partials
  };
  uint16_t kb[kMaxPairs][2][8];  // K-min k-step: B column values (FP16 bits), per pair and head block
  uint32_t qp[8][64];            // q of the unit, per head: FP16 pairs in B-fragment order (odd channels / 16)
  uint32_t qn[8][64];            // q of the unit, per head: FP16 pairs of channels (2c, 2c + 1)
  unsigned long long mask[kLoops];  // presence of the tile's tokens in each sparse loop
  float red[kGroupWarps][8];        // per-warp running max per head (unit-end merge)
  float lsum[kGroupWarps][8];
  float vbs[kGroupWarps][2][8];
  int32_t abort;
};

struct Smem {
  Stage st[kStages];
  GroupSmem grp[kGroups];
  unsigned long long full[kStages];
  unsigned long long empty[kStages];
};
static_assert(sizeof(Smem) <= 227 * 1024, "one block per SM: at most 227 KB of shared memory");

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

// A waiting thread is suspended for at most kSuspendNs per try (the default,
// system-dependent limit let a waiter sleep well past the phase completion).
constexpr uint32_t kSuspendNs = 200;

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendNs)
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

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit values held one row pair per thread.
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ uint32_t h2u(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 u2h(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// ---------------------------------------------------------------- producer
//
// A group's two producer warps take alternate tiles (warp p fills stage p of
// the group's two), so that one warp's copy set-up overlaps the other's. Lane
// 8 j + c serves loop j with one 1-D bulk copy: c = 0 the K code block, 1 the
// V code block (up to 4 KB each), 2 and 3 the K min and scale rows of the
// tile's groups (256 B per group each), 4 and 5 the V min and scale rows
// (4 B per row, in whole 16-byte units), 6 a sparse loop's index slice. All
// per-tile arithmetic - rows, groups, pairs, sizes, the stage's expected byte
// count - comes before the wait for a free stage; after it the warp only
// issues the copies and writes the metadata, and lane 0 arrives. (Issuing the
// small planes as many 16-byte asynchronous copies instead cost the producer
// warp thousands of cycles per tile, which the consumers waited for.)

template <int DEPTH>
__device__ void producer(const AttnArgs& a, Smem& S, int grp, int pw, long long s0, long long e0, int lane) {
  const int j = lane >> 3, c = lane & 7;  // this lane's loop and slot within it
  int b = request_of(a.prefix, a.n_requests, s0);
  long long us = 0, ue = -1;  // current unit's tile range
  int h = 0, T = 0, unit = -1, nsink = 0;
  int nr = 0, kgr = 0, rs = 0, gs = 0;  // this lane's loop: stored rows, tile K groups, plane strides
  const int32_t* act = nullptr;
  const int32_t* dir = nullptr;
  const uint8_t* codes = nullptr;  // the code plane of this lane (c < 2)
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
        act = L.active_idx;
        dir = L.tile_dir;
        codes = c == 0 ? L.k_codes : L.v_codes;
        kmn = reinterpret_cast<const uint8_t*>(L.k_mins);
        ksc = reinterpret_cast<const uint8_t*>(L.k_scales);
        vmn = reinterpret_cast<const uint8_t*>(L.v_mins);
        vsc = reinterpret_cast<const uint8_t*>(L.v_scales);
      }
    }
    // the group's two producer warps take alternate tiles: warp pw fills stage pw
    if (int(it & 1) != pw) continue;
    const int k = int(x - us);
    int c0 = 0, c1 = 0;
    if (j < DEPTH) {
      if (act == nullptr) {
        c0 = k * KVQ_TILE;
        c1 = min(k * KVQ_TILE + KVQ_TILE, T);
      } else {
        c0 = __ldg(dir + k);
        c1 = __ldg(dir + k + 1);
      }
    }
    // this lane's loop: rows of the tile, K groups, pairs
    bool bad = false;
    int n = 0, g0 = 0, ngrp = 0;
    const bool kt = kgr > 0;
    if (j < DEPTH) {
      if (c0 < 0 || c1 > nr || c0 > c1 || c1 - c0 > KVQ_TILE || (j == 0 && act != nullptr)) {
        bad = true;
        c0 = c1 = 0;
      }
      n = c1 - c0;
      g0 = kt ? k : c0 / kG;
      ngrp = n > 0 ? (kt ? 1 : (c1 - 1) / kG - g0 + 1) : 0;
    }
    int pbase = 0, np = 0;  // pairs of the earlier loops, of all loops
#pragma unroll
    for (int jj = 0; jj < DEPTH; ++jj) {
      const int gj = __shfl_sync(0xffffffffu, ngrp, 8 * jj);
      pbase += jj < j ? gj : 0;
      np += gj;
    }
    if (np > kMaxPairs) {  // cannot happen for a table the plan accepted (loop 1 dense); refuse the tile's rows
      bad = true;
      ngrp = 0;
      np = 0;
    }
    const bool live = j < DEPTH && ngrp > 0;
    const long long hr = (long long)h * rs + c0;  // first stored row of this head
    // this lane's copy: source, size (16-byte aligned and rounded, as every plane starts on a 16-byte boundary)
    const long long voff = hr * 4, vlo = voff & ~15LL;
    const long long ioff = (long long)c0 * 4, ilo = ioff & ~15LL;
    const int vrem = int((voff - vlo) / 2), irem = int((ioff - ilo) / 4);
    uint32_t bytes = 0;
    const uint8_t* src = nullptr;
    if (live) {
      const long long kb = ((long long)h * gs + g0) * kD * 2;
      const uint32_t vbytes = uint32_t(((voff + (long long)n * 4 + 15) & ~15LL) - vlo);
      switch (c) {
        case 0:
        case 1: bytes = uint32_t(n * kRowBytes); src = codes + hr * kRowBytes; break;
        case 2: bytes = uint32_t(ngrp * kD * 2); src = kmn + kb; break;
        case 3: bytes = uint32_t(ngrp * kD * 2); src = ksc + kb; break;
        case 4: bytes = vbytes; src = vmn + vlo; break;
        case 5: bytes = vbytes; src = vsc + vlo; break;
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
        LM[0] = ngrp > 0 ? n : 0;
        LM[1] = kt ? k * kG : c0;
        LM[2] = g0;
        LM[3] = ngrp;
        LM[4] = vrem;
        LM[5] = irem;
        LM[6] = act != nullptr;
        LM[7] = pbase;
        if (bad) atomicOr(a.err, 4);
      } else if (c == 1 || c == 2) {
        if (c - 1 < ngrp) M[8 + pbase + c - 1] = (j << 1) | (c - 1);
      }
    }
    // the single expected arrival releases the metadata (ordered after every
    // lane's writes by the warp barrier)
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.full[s]);
  }
}

// ---------------------------------------------------------------- consumers

struct UnitState {
  float m[2];       // running max per head slot (log2 units)
  float l[2];       // partial sums of exp2 of this thread's tokens, per head slot
  float vb[2][2];   // V-min terms: [V group][head slot]
  float acc[8][4];  // PV accumulators: m-tile (V group, channel pair) x (rows g, g + 8) x (columns 2q, 2q + 1)
};

struct UnitInfo {
  int unit, b, h, whole;
};

// Head of slot e of a thread with lane quad index q: with eight query heads a
// thread holds heads q and q + 4, else head q.
template <bool G8>
__device__ __forceinline__ int head_of(int q, int e) {
  return G8 ? q + 4 * e : q;
}

// q of the unit into the two FP16 layouts the prep reads.
__device__ void load_unit_query(const AttnArgs& a, GroupSmem& G, int b, int h, int gt) {
  for (int i = gt; i < 8 * 64; i += kGroupThreads) {
    const int hh = i >> 6, c = i & 63;
    const uint16_t* qr = a.q + ((long long)b * a.Hq + (long long)h * a.g + hh) * kD;
    auto qv = [&](int d) { return hh < a.g ? bf16_bits_to_f32(qr[d]) : 0.0f; };
    G.qn[hh][c] = h2u(__floats2half2_rn(qv(2 * c), qv(2 * c + 1)));
    // B-fragment order: c = 16 q' + 4 i + r over channels 32 q' + 8 i + {0, 4 | 1, 5 | 2, 6 | 3, 7}, the odd
    // channels divided by 16 (their codes carry 2^-20)
    const int base = 32 * (c >> 4) + 8 * ((c >> 2) & 3), r = c & 3;
    const int lo = base + (r >> 1) * 2 + (r & 1);
    const float f = (r & 1) ? 0.0625f : 1.0f;
    G.qp[hh][c] = h2u(__floats2half2_rn(qv(lo) * f, qv(lo + 4) * f));
  }
}

// Per-tile preparation by the group: the QK^T B fragments of every (loop, K
// group) pair, the K-min k-step columns (warp 0, one MMA chain over the pairs'
// min rows), and the presence masks of the sparse loops (warps 1..3).
template <int DEPTH, bool G8>
__device__ void prep_tile(const AttnArgs& a, GroupSmem& Gs, const Stage& st, int npairs, int t0, int gt, int w,
                          int lane) {
  constexpr int kHeads = G8 ? 8 : 4;
  const int items = npairs * 16 * kHeads;
  for (int it = gt; it < items; it += kGroupThreads) {
    const int p = it / (16 * kHeads), r = it % (16 * kHeads);
    const int hd = r >> 4, qq = (r >> 2) & 3, i = r & 3;
    const int pj = st.meta[8 + p];
    const uint4 sv = *reinterpret_cast<const uint4*>(&st.l[pj >> 1].ksc[(pj & 1) * kD + 32 * qq + 8 * i]);
    const uint4 qv = *reinterpret_cast<const uint4*>(&Gs.qp[hd][16 * qq + 4 * i]);
    const uint32_t sp[4] = {__byte_perm(sv.x, sv.z, 0x5410), __byte_perm(sv.x, sv.z, 0x7632),
                            __byte_perm(sv.y, sv.w, 0x5410), __byte_perm(sv.y, sv.w, 0x7632)};
    const uint32_t qa[4] = {qv.x, qv.y, qv.z, qv.w};
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 hv = __hmul2(u2h(qa[k]), u2h(sp[k]));               // RN16(q * s)
      hi[k] = h2u(hv);
      lo[k] = h2u(__hfma2(u2h(qa[k]), u2h(sp[k]), __hneg2(hv)));  // RN16(q * s - hi)
    }
    const int blk = hd >> 2, hh = hd & 3;
    Gs.qf[p][blk][i][8 * hh + qq] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    Gs.qf[p][blk][i][8 * hh + 4 + qq] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  const int g = lane >> 2, q = lane & 3;
  if (w == 0) {
    // K-min terms q . mK of every pair: rows = pairs, columns = heads, K = channels
    float cc[2][4] = {};  // two accumulation chains (even and odd k-steps)
    const bool live = g < npairs;
    const int pj = live ? st.meta[8 + g] : 0;
    const uint16_t* mrow = &st.l[pj >> 1].kmin[(pj & 1) * kD];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint32_t a0 = live ? *reinterpret_cast<const uint32_t*>(mrow + 16 * s + 2 * q) : 0u;
      const uint32_t a2 = live ? *reinterpret_cast<const uint32_t*>(mrow + 16 * s + 2 * q + 8) : 0u;
      mma16816(cc[s & 1], a0, 0u, a2, 0u, Gs.qn[g][8 * s + q], Gs.qn[g][8 * s + q + 4]);
    }
    const float c[2] = {cc[0][0] + cc[1][0], cc[0][1] + cc[1][1]};
    if (live) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int head = 2 * q + e;
        const float v = c[e] * 0.0009765625f;  // 2^-10: with A = 2^-14 the product carries 2^-24
        const __half hv = __float2half_rn(v);
        const __half lv = __float2half_rn(v - __half2float(hv));
        Gs.kb[g][head >> 2][2 * (head & 3)] = __half_as_ushort(hv);
        Gs.kb[g][head >> 2][2 * (head & 3) + 1] = __half_as_ushort(lv);
      }
    }
  } else if (w < DEPTH) {
    // presence of the tile's tokens in sparse loop w, from its staged index
    // slice (at most 64 entries: two per lane, OR-reduced over the warp)
    const int4 la = *reinterpret_cast<const int4*>(&st.meta[16 + 8 * w]);
    const int4 lb = *reinterpret_cast<const int4*>(&st.meta[20 + 8 * w]);
    if (lb.z) {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int i0 = 0; i0 < KVQ_TILE; i0 += 32) {
        const int i = i0 + lane;
        const int u = i < la.x ? st.l[w].idx[lb.y + i] - t0 : -1;
        if (u >= 0 && u < 32) lo |= 1u << u;
        if (u >= 32 && u < KVQ_TILE) hi |= 1u << (u - 32);
      }
      lo = __reduce_or_sync(0xffffffffu, lo);
      hi = __reduce_or_sync(0xffffffffu, hi);
      if (lane == 0) Gs.mask[w] = (unsigned long long)hi << 32 | lo;
    }
  }
}

// Writes the unit's result: output rows (whole unit) or the group's partial
// slot. The four warps' online-softmax states are merged: each warp rescales
// its sums by exp2(m_warp - m_group) before they are added. Even channels
// carry 2^-24 and odd ones 2^-20 from the subnormal codes.
template <bool G8>
__device__ void finish_unit(const AttnArgs& a, GroupSmem& G, UnitState& U, const UnitInfo& M, int grp, int vcta,
                            int w, int lane) {
  constexpr int kSlots = G8 ? 2 : 1;
  const int gt = w * 32 + lane;
  const int g = lane >> 2, q = lane & 3;
  if (g == 0) {
    G.red[w][q] = U.m[0];
    G.red[w][q + 4] = G8 ? U.m[1] : -INFINITY;
  }
  group_sync(grp);
  float sc[2] = {0.f, 0.f};
#pragma unroll
  for (int e = 0; e < kSlots; ++e) {
    const int hh = head_of<G8>(q, e);
    const float mg = fmaxf(fmaxf(G.red[0][hh], G.red[1][hh]), fmaxf(G.red[2][hh], G.red[3][hh]));
    sc[e] = (mg == -INFINITY || U.m[e] == -INFINITY) ? 0.f : exp2f(U.m[e] - mg);
    float l = U.l[e] * sc[e], v0 = U.vb[0][e] * sc[e], v1 = U.vb[1][e] * sc[e];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l += __shfl_xor_sync(0xffffffffu, l, off);
      v0 += __shfl_xor_sync(0xffffffffu, v0, off);
      v1 += __shfl_xor_sync(0xffffffffu, v1, off);
    }
    if (g == 0) {
      G.lsum[w][hh] = l;
      G.vbs[w][0][hh] = v0;
      G.vbs[w][1][hh] = v1;
    }
  }
  const float kLo = 16777216.0f, kHi = 1048576.0f;  // 2^24, 2^20
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const float* c = U.acc[mt];
    if (G8) {  // m-tile (vg, e) = 4 vg + e: rows 64 vg + 8 g + 2e (even) and + 1 (odd); heads q, q + 4
      const int ch = 64 * (mt >> 2) + 8 * g + 2 * (mt & 3);
      G.fin[w][ch][q] = c[0] * sc[0] * kLo;
      G.fin[w][ch][q + 4] = c[1] * sc[1] * kLo;
      G.fin[w][ch + 1][q] = c[2] * sc[0] * kHi;
      G.fin[w][ch + 1][q + 4] = c[3] * sc[1] * kHi;
    } else {  // m-tile e: rows 16 g + 2e (even) and + 1 (odd), V group g >> 2; head q
      const int ch = 16 * g + 2 * mt;
      const bool vg1 = g >= 4;
      G.fin[w][ch][q] = (vg1 ? c[1] : c[0]) * sc[0] * kLo;
      G.fin[w][ch + 1][q] = (vg1 ? c[3] : c[2]) * sc[0] * kHi;
    }
  }
  group_sync(grp);
  const int gq = a.g;
  float* slot = a.partials + (size_t)(vcta + M.unit) * kSlotFloats;
  for (int i = gt; i < gq * kD; i += kGroupThreads) {
    const int hh = i / kD, d = i % kD, vg = d >> 6;
    const float lt = G.lsum[0][hh] + G.lsum[1][hh] + G.lsum[2][hh] + G.lsum[3][hh];
    const float vb = G.vbs[0][vg][hh] + G.vbs[1][vg][hh] + G.vbs[2][vg][hh] + G.vbs[3][vg][hh];
    const float o = (G.fin[0][d][hh] + G.fin[1][d][hh]) + (G.fin[2][d][hh] + G.fin[3][d][hh]) + vb;
    const float mx = fmaxf(fmaxf(G.red[0][hh], G.red[1][hh]), fmaxf(G.red[2][hh], G.red[3][hh]));
    if (M.whole) {
      a.out[((long long)M.b * a.Hq + (long long)M.h * gq + hh) * kD + d] = o / lt;
      if (d == 0) a.stats[(long long)M.b * a.Hq + (long long)M.h * gq + hh] = make_float2(mx, lt);
    } else {
      slot[2 * kMaxG + hh * kD + d] = o;
      if (d == 0) {
        slot[kMaxG + hh] = lt;
        slot[hh] = mx;
      }
    }
  }
  group_sync(grp);
}

// kSp: the sparse-decode branches (key masks of a later loop; every logit of a
// reference pass), in an instantiation of their own.
template <int DEPTH, bool G8, bool kSp>
__device__ void consumer(const AttnArgs& a, Smem& S, int grp, int vcta, long long s0, long long e0) {
  constexpr int kSlots = G8 ? 2 : 1;
  const int gt = threadIdx.x - grp * kGroupThreads;  // thread within the group
  const int w = gt >> 5, lane = gt & 31;
  const int g = lane >> 2, q = lane & 3;
  const int gq = a.g;
  const float lsc = a.scale * kLog2e * 16777216.0f;  // the logits carry 2^-24
  GroupSmem& Gs = S.grp[grp];
  const uint32_t lowA = (1u << g) - 1u, lowC = (1u << (g + 8)) - 1u;  // slice tokens before g, g + 8
  // PV takes the warp's 16 tokens in the order t(kk) = s(kk) for kk < 8 and s(kk - 8) + 8 beyond,
  // s(x) = x ^ ((x >> 1) & 1): the four rows that the q lanes load for one A register (rows 2q of
  // the slice in plain order, all 128 bytes apart, so in the same banks) then alternate between the
  // two 64-byte halves of the bank line (rows 0, 3, 4, 7 and 1, 2, 5, 6). B takes P' of the same
  // tokens: lane group g holds the p of token s(g) (a shuffle from lane group s(g), s being its own
  // inverse), which the transposition turns into the rows of tokens s(2q), s(2q + 1).
  const int gs = g ^ ((g >> 1) & 1);
  const uint32_t lowAs = (1u << gs) - 1u, lowCs = (1u << (gs + 8)) - 1u;  // slice tokens before s(g), s(g) + 8
  uint32_t lowP[4];  // slice tokens before s(2q), s(2q + 1), s(2q) + 8, s(2q + 1) + 8
#pragma unroll
  for (int k = 0; k < 4; ++k) lowP[k] = (1u << (((2 * q + (k & 1)) ^ (q & 1)) + 8 * (k >> 1))) - 1u;
  UnitState U;
  int cur_unit = -1;
  UnitInfo Mprev = {-1, 0, 0, 0};
  long long it = 0;

  for (long long x = s0; x < e0; ++x, ++it) {
    const int s = grp * kStagesPerGroup + int(it & 1);
    const uint32_t ph = uint32_t((it >> 1) & 1);
    if (!mbar_wait(&S.full[s], ph) && lane == 0) Gs.abort = 1;
    // every warp is past the previous tile (its fragments may be rewritten) and
    // all agree on whether to go on
    group_sync(grp);
    if (Gs.abort) {
      if (gt == 0) atomicOr(a.err, 8);
      return;
    }
    const Stage& st = S.st[s];
    const int4 m0 = *reinterpret_cast<const int4*>(&st.meta[0]);
    const int4 m1 = *reinterpret_cast<const int4*>(&st.meta[4]);
    const int unit = m0.x, t0 = m0.w, nvalid = m1.x, npairs = m1.z, tfirst = m1.w;
    if (unit != cur_unit) {
      if (cur_unit >= 0) finish_unit<G8>(a, Gs, U, Mprev, grp, vcta, w, lane);
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
    }
    // sparse decode, later loop: the selection bits of the warp's 16 tokens for this thread's query
    // heads (one mask word covers them), loaded here so that their latency overlaps the tile's QK;
    // a request longer than the masks cover (the sparse path refuses it) selects nothing here
    uint32_t selw[2] = {0u, 0u};
    if (kSp && a.sel_mask != nullptr) {
      const int tb = t0 + 16 * w;
      const bool in = (tb >> 5) < a.mask_words;
#pragma unroll
      for (int e = 0; e < kSlots; ++e) {
        const int hh = head_of<G8>(q, e);
        if (in && hh < gq)
          selw[e] = __ldg(a.sel_mask + ((long long)Mprev.b * a.Hq + (long long)Mprev.h * gq + hh) * a.mask_words +
                          (tb >> 5)) >> (tb & 31);
      }
    }
    prep_tile<DEPTH, G8>(a, Gs, st, npairs, t0, gt, w, lane);
    group_sync(grp);  // fragments, K-min columns and presence masks ready

    // ---- QK^T of the warp's 16 tokens [16w, 16w + 16) over every loop, in the
    // accumulator layout: C[slot][chain] = {(token g, hi), (g, lo), (g + 8, hi), (g + 8, lo)};
    // independent accumulation chains (four, or two with eight query heads: k-step (i, hf)
    // goes to chain 2 (i & 1) + hf, or hf), summed after the last loop
    constexpr int kChains = G8 ? 2 : 4;
    float C[kSlots][kChains][4];
#pragma unroll
    for (int e = 0; e < kSlots; ++e)
#pragma unroll
      for (int ch = 0; ch < kChains; ++ch) C[e][ch][0] = C[e][ch][1] = C[e][ch][2] = C[e][ch][3] = 0.f;
    // per loop: presence of the warp's 16 tokens and the first stored row of its slice, for every
    // loop before the contractions (a dense loop stores the tile's first nrows tokens at rows
    // 0 .. nrows - 1; a sparse loop's presence mask was built with the fragments; the branch-free
    // form lets the loops' loads issue together)
    uint32_t pbits[DEPTH];
    int prb[DEPTH];
#pragma unroll
    for (int j = 0; j < DEPTH; ++j) {
      const int nrows = st.meta[16 + 8 * j], sparse = st.meta[22 + 8 * j];
      const unsigned long long mk = Gs.mask[j];  // stale for a dense loop, and then unused
      const int cnt = max(0, min(16, nrows - 16 * w));
      const uint32_t dense_bits = cnt >= 16 ? 0xFFFFu : ((1u << cnt) - 1u);
      pbits[j] = nrows == 0 ? 0u : (sparse ? uint32_t(mk >> (16 * w)) & 0xFFFFu : dense_bits);
      prb[j] = nrows == 0 ? 0 : (sparse ? __popcll(mk & ((1ull << (16 * w)) - 1ull)) : 16 * w);
    }
#pragma unroll
    for (int j = 0; j < DEPTH; ++j) {
      const uint32_t bits = pbits[j];
      if (bits == 0) continue;
      const int rb = prb[j];
      const int4 la = *reinterpret_cast<const int4*>(&st.meta[16 + 8 * j]);
      const int4 lb = *reinterpret_cast<const int4*>(&st.meta[20 + 8 * j]);
      const int c0 = la.y, g0 = la.z, ngrp = la.w, pbase = lb.w;
      // stored rows of tokens g and g + 8: the first row of the warp's slice plus the token's rank
      // among the slice's stored tokens (a dense slice stores them all, so the rank is the token);
      // an absent token gets a row index <= 64, inside the stage, whose codes its zero A row ignores
      const bool pa = (bits >> g) & 1, pc = (bits >> (g + 8)) & 1;
      const int ra = rb + __popc(bits & lowA), rc = rb + __popc(bits & lowC);
      const uint4 wa = *reinterpret_cast<const uint4*>(&st.l[j].kc[ra * kRowBytes + 16 * q]);
      const uint4 wb = *reinterpret_cast<const uint4*>(&st.l[j].kc[rc * kRowBytes + 16 * q]);
      const uint32_t wA[4] = {wa.x, wa.y, wa.z, wa.w}, wB[4] = {wb.x, wb.y, wb.z, wb.w};
      // K groups of the warp's rows: one for dense loops and tile grouping; the rows of a
      // compact-grouped sparse loop may span two, and each pass then keeps its group's tokens
      int ga = 0, gb = 0, sa = 0, sc = 0;
      if (ngrp > 1) {
        ga = ((c0 + rb) >> 6) - g0;
        gb = ((c0 + rb + __popc(bits) - 1) >> 6) - g0;
        sa = ((c0 + ra) >> 6) - g0;
        sc = ((c0 + rc) >> 6) - g0;
      }
      auto pass = [&](int G) {
        const bool ka = pa && sa == G, kc = pc && sc == G;
        const uint32_t la_ = ka ? kLoMask : 0u, ha_ = ka ? kHiMask : 0u;
        const uint32_t lc_ = kc ? kLoMask : 0u, hc_ = kc ? kHiMask : 0u;
        const int pair = pbase + G;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t xa = wA[i], xb = wB[i], ya = xa >> 8, yb = xb >> 8;
          const uint32_t a0 = xa & la_, a1 = xb & lc_, a2 = xa & ha_, a3 = xb & hc_;
          const uint32_t a4 = ya & la_, a5 = yb & lc_, a6 = ya & ha_, a7 = yb & hc_;
          const int ch = kChains == 4 ? 2 * (i & 1) : 0;
#pragma unroll
          for (int e = 0; e < kSlots; ++e) {
            const uint4 bq = Gs.qf[pair][e][i][lane];
            mma16816(C[e][ch], a0, a1, a2, a3, bq.x, bq.y);
            mma16816(C[e][ch + 1], a4, a5, a6, a7, bq.z, bq.w);
          }
        }
        // the K-min k-step: A = 2^-14 at k = 0 for a stored token of this group
        const uint32_t kA = (q == 0 && ka) ? kKbA : 0u, kC = (q == 0 && kc) ? kKbA : 0u;
#pragma unroll
        for (int e = 0; e < kSlots; ++e) {
          const uint32_t kb0 = q == 0 ? uint32_t(Gs.kb[pair][e][g]) : 0u;
          mma16816(C[e][0], kA, kC, 0u, 0u, kb0, 0u);
        }
      };
      pass(ga);
      if (gb != ga) pass(gb);
    }

    // ---- logits in log2 units, this warp's max per head, online softmax
    const int tA = 16 * w + g, tC = tA + 8;
    const bool vA = tA < nvalid && tA >= tfirst, vC = tC < nvalid && tC >= tfirst;
    float pA[2] = {0.f, 0.f}, pC[2] = {0.f, 0.f}, al[2] = {1.f, 1.f};
#pragma unroll
    for (int e = 0; e < kSlots; ++e) {
      const bool hok = head_of<G8>(q, e) < gq;
      float c4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        c4[k] = C[e][0][k] + C[e][1][k];
        if (kChains == 4) c4[k] += C[e][2][k] + C[e][3][k];
      }
      float sA = (vA && hok) ? (c4[0] + c4[1]) * lsc : -INFINITY;
      float sC = (vC && hok) ? (c4[2] + c4[3]) * lsc : -INFINITY;
      if (kSp && a.logits != nullptr) {  // sparse decode reference pass: every logit, for the selection
        float* lr = a.logits + ((long long)Mprev.b * a.Hq + (long long)Mprev.h * gq + head_of<G8>(q, e)) *
                                   a.logit_stride;
        if (vA && hok && t0 + tA < a.logit_stride) lr[t0 + tA] = sA;
        if (vC && hok && t0 + tC < a.logit_stride) lr[t0 + tC] = sC;
      }
      if (kSp && a.sel_mask != nullptr) {  // sparse decode later loop: only the query head's selected keys
        if (!((selw[e] >> g) & 1u)) sA = -INFINITY;
        if (!((selw[e] >> (g + 8)) & 1u)) sC = -INFINITY;
      }
      float mt = fmaxf(sA, sC);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float mn = fmaxf(U.m[e], mt);
      al[e] = (U.m[e] == -INFINITY) ? 0.f : exp2f(U.m[e] - mn);
      U.m[e] = mn;
      pA[e] = sA == -INFINITY ? 0.f : exp2f(sA - mn);
      pC[e] = sC == -INFINITY ? 0.f : exp2f(sC - mn);
      U.l[e] = U.l[e] * al[e] + (pA[e] + pC[e]);
    }
    if (__any_sync(0xffffffffu, al[0] != 1.f || al[1] != 1.f)) {
#pragma unroll
      for (int vg = 0; vg < 2; ++vg) {
        U.vb[vg][0] *= al[0];
        U.vb[vg][1] *= al[1];
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        U.acc[mt][0] *= al[0];
        U.acc[mt][1] *= G8 ? al[1] : al[0];
        U.acc[mt][2] *= al[0];
        U.acc[mt][3] *= G8 ? al[1] : al[0];
      }
    }

    // ---- PV over every loop (tokens s(g), s(g) + 8 in this lane group's B rows)
    float pAs[2], pCs[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      pAs[e] = __shfl_sync(0xffffffffu, pA[e], 4 * gs + q);
      pCs[e] = __shfl_sync(0xffffffffu, pC[e], 4 * gs + q);
    }
#pragma unroll
    for (int j = 0; j < DEPTH; ++j) {
      const uint32_t bits = pbits[j];
      if (bits == 0) continue;
      const int rb = prb[j];
      const int vrem = st.meta[16 + 8 * j + 4];
      const bool pa = (bits >> gs) & 1, pc = (bits >> (gs + 8)) & 1;
      const int ra = rb + __popc(bits & lowAs), rc = rb + __popc(bits & lowCs);
      // V params of tokens s(g), s(g) + 8 ({group 0, group 1} pairs), P' = RN16(p * sV) and the V-min
      // terms (a token without a stored row reads nothing: its staged slot may hold stale bits)
      const uint32_t sva = pa ? *reinterpret_cast<const uint32_t*>(&st.l[j].vsc[vrem + 2 * ra]) : 0u;
      const uint32_t svc = pc ? *reinterpret_cast<const uint32_t*>(&st.l[j].vsc[vrem + 2 * rc]) : 0u;
      const float2 mva =
          __half22float2(u2h(pa ? *reinterpret_cast<const uint32_t*>(&st.l[j].vmin[vrem + 2 * ra]) : 0u));
      const float2 mvc =
          __half22float2(u2h(pc ? *reinterpret_cast<const uint32_t*>(&st.l[j].vmin[vrem + 2 * rc]) : 0u));
      float qa[2], qc[2];  // p of the slots, zero for a token without a row in this loop
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        qa[e] = pa ? pAs[e] : 0.f;
        qc[e] = pc ? pCs[e] : 0.f;
      }
      // A: V codes of tokens s(2q), s(2q + 1), s(2q) + 8, s(2q + 1) + 8 (a token without a row
      // reads a valid row against a zero P')
      const uint8_t* vbase = &st.l[j].vc[0];
      int ro[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) ro[k] = (rb + __popc(bits & lowP[k])) * kRowBytes;
      if (G8) {
        // B per V group: columns 2q, 2q + 1 = heads q, q + 4; thread g takes word 8 vg + g of each
        // row (channels 64 vg + 8 g .. + 7); m-tile (vg, e) has rows 8g + 2e and 8g + 2e + 1
        uint32_t B[2][2];
#pragma unroll
        for (int vg = 0; vg < 2; ++vg) {
          const __half2 sa2 = vg == 0 ? __low2half2(u2h(sva)) : __high2half2(u2h(sva));
          const __half2 sc2 = vg == 0 ? __low2half2(u2h(svc)) : __high2half2(u2h(svc));
          B[vg][0] = transpose8x8(h2u(__hmul2(__floats2half2_rn(qa[0], qa[1]), sa2)));
          B[vg][1] = transpose8x8(h2u(__hmul2(__floats2half2_rn(qc[0], qc[1]), sc2)));
        }
        U.vb[0][0] = fmaf(qa[0], mva.x, fmaf(qc[0], mvc.x, U.vb[0][0]));
        U.vb[1][0] = fmaf(qa[0], mva.y, fmaf(qc[0], mvc.y, U.vb[1][0]));
        U.vb[0][1] = fmaf(qa[1], mva.x, fmaf(qc[1], mvc.x, U.vb[0][1]));
        U.vb[1][1] = fmaf(qa[1], mva.y, fmaf(qc[1], mvc.y, U.vb[1][1]));
#pragma unroll
        for (int vg = 0; vg < 2; ++vg) {
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vbase + ro[0] + 4 * (8 * vg + g));
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vbase + ro[1] + 4 * (8 * vg + g));
          const uint32_t w2 = *reinterpret_cast<const uint32_t*>(vbase + ro[2] + 4 * (8 * vg + g));
          const uint32_t w3 = *reinterpret_cast<const uint32_t*>(vbase + ro[3] + 4 * (8 * vg + g));
          const uint32_t xv[2] = {__byte_perm(w0, w1, 0x5410), __byte_perm(w0, w1, 0x7632)};
          const uint32_t yv[2] = {__byte_perm(w2, w3, 0x5410), __byte_perm(w2, w3, 0x7632)};
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const uint32_t x = xv[hb], y = yv[hb], xs = x >> 8, ys = y >> 8;
            mma16816(U.acc[4 * vg + 2 * hb], x & kLoMask, x & kHiMask, y & kLoMask, y & kHiMask, B[vg][0],
                     B[vg][1]);
            mma16816(U.acc[4 * vg + 2 * hb + 1], xs & kLoMask, xs & kHiMask, ys & kLoMask, ys & kHiMask,
                     B[vg][0], B[vg][1]);
          }
        }
      } else {
        // one B for both V groups: columns 2q, 2q + 1 = head q with V group 0, 1 (each output row
        // keeps the column of its channel's group); thread g takes bytes 8g .. 8g + 7 of each row
        // (channels 16 g .. 16 g + 15); m-tile e has rows 16g + 2e and 16g + 2e + 1
        const uint32_t B0 = transpose8x8(h2u(__hmul2(__float2half2_rn(qa[0]), u2h(sva))));
        const uint32_t B1 = transpose8x8(h2u(__hmul2(__float2half2_rn(qc[0]), u2h(svc))));
        U.vb[0][0] = fmaf(qa[0], mva.x, fmaf(qc[0], mvc.x, U.vb[0][0]));
        U.vb[1][0] = fmaf(qa[0], mva.y, fmaf(qc[0], mvc.y, U.vb[1][0]));
        const uint2 u0 = *reinterpret_cast<const uint2*>(vbase + ro[0] + 8 * g);
        const uint2 u1 = *reinterpret_cast<const uint2*>(vbase + ro[1] + 8 * g);
        const uint2 u2 = *reinterpret_cast<const uint2*>(vbase + ro[2] + 8 * g);
        const uint2 u3 = *reinterpret_cast<const uint2*>(vbase + ro[3] + 8 * g);
#pragma unroll
        for (int hw = 0; hw < 2; ++hw) {
          const uint32_t w0 = hw ? u0.y : u0.x, w1 = hw ? u1.y : u1.x, w2 = hw ? u2.y : u2.x, w3 = hw ? u3.y : u3.x;
          const uint32_t xv[2] = {__byte_perm(w0, w1, 0x5410), __byte_perm(w0, w1, 0x7632)};
          const uint32_t yv[2] = {__byte_perm(w2, w3, 0x5410), __byte_perm(w2, w3, 0x7632)};
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const uint32_t x = xv[hb], y = yv[hb], xs = x >> 8, ys = y >> 8;
            mma16816(U.acc[4 * hw + 2 * hb], x & kLoMask, x & kHiMask, y & kLoMask, y & kHiMask, B0, B1);
            mma16816(U.acc[4 * hw + 2 * hb + 1], xs & kLoMask, xs & kHiMask, ys & kLoMask, ys & kHiMask, B0, B1);
          }
        }
      }
    }
    // release the stage: every warp of the group is done reading it
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
  }
  if (cur_unit >= 0) finish_unit<G8>(a, Gs, U, Mprev, grp, vcta, w, lane);
}

template <int DEPTH, bool G8, bool kSp>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int C = a.n_ctas;  // virtual CTAs: two per block
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kGroupWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the group areas start zeroed: fragment columns of absent query heads stay zero
  for (int i = threadIdx.x; i < int(sizeof(GroupSmem) * kGroups / 16); i += kThreads)
    reinterpret_cast<uint4*>(S.grp)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  wait_prior_grid();  // the plan (tile prefix, error word) is complete and visible from here on
  if (a.dispatch == 1 && (*a.flags & 2)) return;  // the plan found NVFP4 loops: the NVFP4-reading kernel runs
  const long long W = a.prefix[a.n_requests];
  int grp, pw = 0;
  bool producer_warp;
  if (threadIdx.x < kConsumers) {
    grp = threadIdx.x / kGroupThreads;
    producer_warp = false;
  } else {
    const int pwarp = (threadIdx.x - kConsumers) >> 5;
    grp = pwarp / kProducers;
    pw = pwarp % kProducers;
    producer_warp = true;
  }
  const int vcta = kGroups * blockIdx.x + grp;
  const long long s0 = cta_start(vcta, W, C), e0 = cta_start(vcta + 1, W, C);
  if (s0 >= e0) return;
  if (producer_warp) {
    producer<DEPTH>(a, S, grp, pw, s0, e0, threadIdx.x & 31);
    return;
  }
  consumer<DEPTH, G8, kSp>(a, S, grp, vcta, s0, e0);
}

template <int DEPTH, bool G8, bool kSp>
cudaError_t launch_depth(const AttnArgs& a, cudaStream_t stream) {
  const int smem = int(sizeof(Smem));
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_tc_kernel<DEPTH, G8, kSp>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_dependent(attn_tc_kernel<DEPTH, G8, kSp>, dim3(a.n_ctas / kGroups), dim3(kThreads), size_t(smem),
                          stream, a);
}

template <bool kSp>
cudaError_t launch_form(const AttnArgs& a, cudaStream_t stream) {
  switch (a.depth * 2 + (a.g == 8 ? 1 : 0)) {
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

}  // namespace tc_attn

int tc_virtual_ctas_per_block() { return tc_attn::kGroups; }

// The INT4 packed attention (depth <= 4, 1/2/4/8 query heads per KV head),
// dense calls and the sparse-decode passes (key masks, logits); the caller
// refuses requests holding NVFP4 loops in the plan.
cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t stream) {
  using namespace tc_attn;
  const cudaError_t e = (a.sel_mask != nullptr || a.logits != nullptr) ? launch_form<true>(a, stream)
                                                                        : launch_form<false>(a, stream);
  if (e == cudaErrorInvalidValue) return e;
  count_launch();
  return e;
}

}  // namespace kvq
