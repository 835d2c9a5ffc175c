// kvq_attn_tcgen05.cu — decode attention over packed INT4 K/V chains on the
// fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// FlashLoop RFC (vllm-rlt issue #156) §3.2: historical K/V are read at the
// requested depth and reconstructed if compressed, scores scaled by
// 1/sqrt(head_dim); §3.3: optimized readers consume the packed base/residual
// tiles directly during QK/PV, with the affine INT4 group code
// decode = min + scale * code; §5: FP32 mass and accumulation.
//
// Work list, partial slots, plan and merge are those of kvq_attn_common.cuh;
// every block is one CTA of the work split (one block per SM). Selected with
// KVQ_ATTN_TCGEN05; the default INT4 path is the mma.sync form of
// kvq_attn_tc.cu, which is about twice as fast on the decode shapes: there the
// unpacked codes feed the MMAs from registers, while here every code is first
// written to tensor or shared memory, and each tcgen05.mma of these small
// shapes (N = 8..32) costs its issuing warp about 50 cycles.
//
// Codes as FP16 subnormals. A 32-bit word of packed codes holds channels
// 8i .. 8i + 7 of a row (low nibble = even channel). AND-ing it with 0x000F000F
// leaves FP16 pairs n * 2^-24 (channels 8i, 8i + 4); with 0x00F000F0, n * 2^-20
// (8i + 1, 8i + 5); the same on the word shifted right by 8 gives (8i + 2,
// 8i + 6) and (8i + 3, 8i + 7). The tensor cores take these subnormals
// exactly, so a code needs no offset and no conversion.
//
// Per tile (64 tokens of one (request, KV head), all loops to the depth):
//   QK^T  loop j: S_j[t, n] = A_j[t, :] . B_j[:, n], tcgen05.mma kind::f16,
//         M = 64 tokens, K = 128 channels, N = (K group, head, hi | lo); A = the
//         loop's codes in tensor memory (tcgen05.st 16x128b: four threads per
//         token row), zero rows for tokens the loop does not store; B = Q' =
//         q * sK of the tile's K groups of the loop (at most two) as an exact
//         FP16 pair hi + lo (hi = RN16(q s), lo = RN16(q s - hi)), divided by 16
//         on the odd channels (their codes carry 2^-20), in shared memory
//         (K-major, no swizzle). A token reads the columns of its own K group.
//         The K-min terms q . mK are one mma.sync chain per tile, added in FP32.
//   softmax  FP32, log2 domain, one running max per query head for the whole
//         CTA (the PV products of all 64 tokens meet in one accumulator).
//   PV    O^T[m, n] = sum_j sum_t A_j[m, t] * P'_j[t, n], tcgen05.mma kind::f16,
//         M = 128 (channels, in the order the unpack produces them), N = 16 =
//         (head, V group), K = 64 tokens; A = the V codes of loop j as FP16
//         subnormals in shared memory (MN-major: a token's channels are
//         contiguous), B = P' = RN16(p * sV) (MN-major). Two accumulators (loops
//         0, 2 and 1, 3) per tile, folded into FP32 registers with the softmax
//         rescale. The V-min terms are FP32 FMAs.
//
// Warp roles (16 warps). A tcgen05.mma costs its issuing warp about 50 cycles
// whatever the decode shape while the tensor cores take several in flight, and
// every phase of a tile is a chain of dependent steps, so the work is split
// into roles that overlap across tiles, meeting on mbarriers:
//   0..3    softmax: K-min terms, logits from the QK accumulators, running
//           max, P' and the V-min terms (16 tokens per warp);
//   4..7    operands, one tile ahead of the softmax: Q', K codes into tensor
//           memory, then (after the previous tile's PV) its fold into the
//           output registers (one channel row per thread) and the V codes into
//           shared memory;
//   8..11   warp 8 + j issues the QK MMAs of loop j into its own accumulator;
//   12, 13  issue the PV MMAs of loops (0, 2) and (1, 3);
//   14, 15  producers: warp p stages every second 64-token tile into stage p
//           (code blocks by bulk copy, the min/scale planes by 16-byte
//           asynchronous copies), with the tile's per-loop token presence
//           masks computed from the sparse index slices.
// Two softmax results cross from the softmax to the operand warps through
// shared-memory slots per tile parity released by sequence counters (the
// rescale of each tile, and a finished unit's sums). Every wait is bounded
// (2 s on %globaltimer): a wait that runs out sets bit 8 of the error word and
// the warps leave at their next check; the MMA issuers wait (bounded) for
// their MMAs before the tensor memory is freed.
#include <cuda_fp16.h>

#include "kvq_attn_common.cuh"

namespace kvq {
namespace t5_attn {

constexpr int kLoops = 4;
constexpr int kStages = 2;
constexpr int kWarpOperand = 4;
constexpr int kWarpQk = 8;
constexpr int kWarpPv = 12;
constexpr int kWarpProducer = 14;
constexpr int kThreads = 16 * 32;
constexpr int kTmemUsers = kWarpProducer * 32;  // every warp but the producers
constexpr int kMaxPairs = 1 + 2 * (kLoops - 1);  // (loop, K group) pairs of a tile: loop 1 is dense
constexpr int kLoopMeta = 12;
constexpr int kMetaWords = 16 + kLoopMeta * kLoops;
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitNs = 2000000000LL;
constexpr uint32_t kLoMask = 0x000F000Fu;  // even channels: FP16 n * 2^-24
constexpr uint32_t kHiMask = 0x00F000F0u;  // odd channels:  FP16 n * 2^-20
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0;    // A of loop j: columns 64 j .. 64 j + 63
constexpr uint32_t kColS = 256;  // QK accumulator of loop j: columns kColS + 32 j .. (two K groups)
constexpr uint32_t kColO = 384;  // PV accumulators: kColO (loops 0, 2) and kColO + 16 (loops 1, 3)

// Per-tile metadata written by the producer (int32 words):
//   [0] unit  [1] b  [2] h  [3] t0  [4] nvalid  [5] whole  [6] npairs
//   [7] first token of the tile read from the packed chain
//   pair p (7 words from 8): loop index << 1 | group
//   loop j (12 words from 16 + 12 j): [0] stored rows in the tile (0: none)
//       [1] c0 (first stored row; under tile grouping of K, 64 x tile) [2] g0
//       [3] K groups [4] vrem [6] sparse [7] pbase [8], [9] presence mask of
//       the tile's tokens (low, high word)

struct LoopStage {
  uint8_t kc[KVQ_TILE * kRowBytes];
  uint8_t vc[KVQ_TILE * kRowBytes];
  uint16_t kmin[2 * kD];
  uint16_t ksc[2 * kD];
  uint16_t vmin[144];  // 64 rows x 2 groups + 16 B rounding slack
  uint16_t vsc[144];
};
static_assert(sizeof(LoopStage) % 16 == 0, "loop stages keep 16-byte alignment");

struct __align__(128) Stage {
  LoopStage l[kLoops];
  int32_t meta[kMetaWords];
};

// Operand layouts (no swizzle; a core matrix is 8 rows of 16 bytes):
//   bq (loop j): K-major B of QK, element (n, k) at (n/8)*2048 + (k/8)*128 + (n%8)*16 + (k%8)*2
//   va[j]: MN-major A of PV, element (token u, row m) at (m/8)*1024 + (u/8)*128 + (u%8)*16 + (m%8)*2
//   bp[.][j]: MN-major B of PV, element (token u, n) at (n/8)*1024 + (u/8)*128 + (u%8)*16 + (n%8)*2
template <bool G8>
struct Smem {
  static constexpr int kNb = G8 ? 16 : 8;  // QK columns of one K group: n = 2 head + (0 hi | 1 lo)
  // Q' of loop j at element offset bq_off(j): loop 0 is dense (one K group), later loops hold two
  __host__ __device__ static constexpr int bq_off(int j) { return j == 0 ? 0 : (kNb + 2 * kNb * (j - 1)) * kD; }
  uint16_t va[kLoops][KVQ_TILE * kD];
  uint16_t bq[(kNb + 2 * kNb * (kLoops - 1)) * kD];
  uint16_t bp[2][kLoops][KVQ_TILE * 16];  // per tile parity
  Stage st[kStages];
  uint32_t qp[8][64];  // operand warps: q of the unit per head, FP16 pairs in QK k order (odd-channel blocks / 16)
  uint32_t qn[8][64];  // softmax warps: q of the unit per head, FP16 pairs of channels (2c, 2c + 1)
  float kmt[4][kMaxPairs][8];  // per softmax warp: K-min terms per (pair, head)
  float red[4][8];             // per softmax warp: max logit per head of the tile
  float alpha[2][8];           // per tile parity: rescale of the tile's softmax step
  float lsum[2][4][8];         // per tile parity: sums of a finished unit, per softmax warp
  float vbs[2][4][2][8];
  float fm[2][8];              // final max per head
  volatile int32_t alpha_seq;  // alpha of tile i is in place once alpha_seq > i
  volatile int32_t sums_seq;   // the slot of tile i is in place once sums_seq > i
  unsigned long long full[kStages];
  unsigned long long empty[kStages];
  unsigned long long ops;     // the tile's Q' and A operands written (4 arrivals: operand warps)
  unsigned long long sread;   // the QK accumulators read (4 arrivals: softmax warps)
  unsigned long long pready;  // P' written (4 arrivals: softmax warps)
  unsigned long long vready;  // V operands written (4 arrivals: operand warps)
  unsigned long long mbS;     // QK accumulators complete (one commit per loop issuer)
  unsigned long long mbO;     // PV accumulators complete (one commit per PV issuer)
  unsigned long long drain;   // every MMA of the issuers complete (one commit per issuer)
  uint32_t tmem;
  volatile int32_t abort;
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

// Named barriers: 1 = the softmax warps, 2 = the operand warps, 3 = every warp
// that touches tensor memory (before it is freed).
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void operand_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
// bar.sync of group `id` (128 threads) that also returns whether any thread passed v = true.
__device__ __forceinline__ bool group_sync_or(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred pi, po; setp.ne.u32 pi, %1, 0; bar.red.or.pred po, %2, 128, pi; selp.u32 %0, 1, 0, po; }"
      : "=r"(r)
      : "r"(uint32_t(v)), "r"(id)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void tmem_users_sync() { asm volatile("bar.sync 3, %0;" ::"n"(kTmemUsers) : "memory"); }

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: start, leading (along K) and stride (along
// M or N) byte offsets between core matrices, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46);
}

// Instruction descriptor of kind::f16: FP16 A and B, FP32 D, the majors of A
// and B (1 = MN-major), N and M.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// D (tensor memory) [+]= A (tensor memory) * B (shared memory)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// D (tensor memory) [+]= A (shared memory) * B (shared memory)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// The mbarrier completes one phase once every MMA issued before is complete.
__device__ __forceinline__ void mma_commit(unsigned long long* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// 16 lanes x 32 columns: register 2n to lane (base + t/4), column 4n + t%4;
// register 2n + 1 to lane (base + t/4 + 8), the same column.
__device__ __forceinline__ void tmem_st_16x128b_x8(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Thread t: registers 0, 1 from lane (base + t/4), columns 2(t%4), 2(t%4) + 1;
// registers 2, 3 from lane (base + t/4 + 8), the same columns. The values are
// valid after tmem_wait_ld() on them (the load is asynchronous).
__device__ __forceinline__ void tmem_ld_16x256b_x1(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}

// Waits for every tcgen05.ld of the thread; the registers named here (and those
// passed to tmem_touch after it) are read only after the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[4]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3])::"memory");
}
__device__ __forceinline__ void tmem_touch(uint32_t (&r)[4]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3])::"memory");
}

// Thread t: 16 consecutive columns of lane (base + t) (waits for the load).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2u(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 u2h(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// ---------------------------------------------------------------- producer
//
// Warp p fills stage p for every second tile. Lane 8 j + c serves loop j: the
// code blocks go by one 1-D bulk copy per (loop, kind) (lanes c = 0 K, 1 V),
// the small planes (K min/scale rows of the tile's groups, V min/scale rows)
// by 16-byte asynchronous copies spread over the loop's lanes. The presence
// mask of a sparse loop comes from its index slice in global memory (eight
// entries per lane, OR-reduced over the loop's lanes), so the consumers need
// no index data.

__device__ __forceinline__ void copy16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

template <int DEPTH, bool G8>
__device__ void producer(const AttnArgs& a, Smem<G8>& S, int pw, long long s0, long long e0, int lane) {
  const int j = lane >> 3, c = lane & 7;  // this lane's loop and slot within it
  int b = request_of(a.prefix, a.n_requests, s0);
  long long us = 0, ue = -1;
  int h = 0, T = 0, unit = -1, nsink = 0;
  int nr = 0, kgr = 0, rs = 0, gs = 0;
  const int32_t* act = nullptr;
  const int32_t* dir = nullptr;
  const uint8_t* codes = nullptr;
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
    if (int(it % kStages) != pw) continue;
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
    // presence mask of the tile's tokens in this lane's loop (read before the
    // wait for a free stage, so that its latency overlaps it)
    uint32_t mlo = 0, mhi = 0;
    if (j < DEPTH && n > 0) {
      if (act == nullptr) {
        if (c == 0) {
          mlo = n >= 32 ? 0xffffffffu : ((1u << n) - 1u);
          mhi = n >= 64 ? 0xffffffffu : (n > 32 ? ((1u << (n - 32)) - 1u) : 0u);
        }
      } else {
        const int tk0 = k * KVQ_TILE;
        for (int i = c; i < n; i += 8) {
          const int u = __ldg(act + c0 + i) - tk0;
          if (u >= 0 && u < 32) mlo |= 1u << u;
          else if (u >= 32 && u < KVQ_TILE) mhi |= 1u << (u - 32);
        }
      }
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      mlo |= __shfl_xor_sync(0xffffffffu, mlo, off);
      mhi |= __shfl_xor_sync(0xffffffffu, mhi, off);
    }
    if (j < DEPTH && n > 0 && __popc(mlo) + __popc(mhi) != n) bad = true;  // positions outside the tile or repeated
    const int s = pw;
    const uint32_t ph = uint32_t((it / kStages) & 1);
    int ok = 1;
    if (lane == 0 && it >= kStages) ok = mbar_wait(&S.empty[s], ph ^ 1u) ? 1 : 0;
    if (!__shfl_sync(0xffffffffu, ok, 0)) {
      if (lane == 0) atomicOr(a.err, 8);
      return;
    }
    Stage& st = S.st[s];
    int32_t* M = st.meta;
    int pbase = 0, np = 0;
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
    const long long hr = (long long)h * rs + c0;
    const uint32_t bytes = (live && c < 2) ? uint32_t(n * kRowBytes) : 0u;
    uint32_t total = bytes;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
    if (lane == 0) mbar_expect_tx(&S.full[s], total);
    __syncwarp();
    if (bytes > 0) {
      LoopStage& LS = st.l[j];
      asm volatile(
          "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              smem_addr(c == 0 ? (void*)LS.kc : (void*)LS.vc)),
          "l"(codes + hr * kRowBytes), "r"(bytes), "r"(smem_addr(&S.full[s]))
          : "memory");
    }
    int vrem = 0;
    if (live) {
      LoopStage& LS = st.l[j];
      const long long kb = ((long long)h * gs + g0) * kD * 2;
      const int nk = ngrp * (kD * 2 / 16);
      const long long voff = hr * 4, vlo = voff & ~15LL;
      const int nv = int((((voff + (long long)n * 4 + 15) & ~15LL) - vlo) / 16);
      vrem = int((voff - vlo) / 2);
      const int ntot = 2 * nk + 2 * nv;
      for (int t = c; t < ntot; t += 8) {
        if (t < nk) {
          copy16(reinterpret_cast<uint8_t*>(LS.kmin) + 16 * t, kmn + kb + 16 * t);
        } else if (t < 2 * nk) {
          copy16(reinterpret_cast<uint8_t*>(LS.ksc) + 16 * (t - nk), ksc + kb + 16 * (t - nk));
        } else if (t < 2 * nk + nv) {
          copy16(reinterpret_cast<uint8_t*>(LS.vmin) + 16 * (t - 2 * nk), vmn + vlo + 16 * (t - 2 * nk));
        } else {
          copy16(reinterpret_cast<uint8_t*>(LS.vsc) + 16 * (t - 2 * nk - nv), vsc + vlo + 16 * (t - 2 * nk - nv));
        }
      }
    }
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(&S.full[s])) : "memory");
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
      int32_t* LM = M + 16 + kLoopMeta * j;
      if (c == 0) {
        LM[0] = ngrp > 0 ? n : 0;
        LM[1] = kt ? k * kG : c0;
        LM[2] = g0;
        LM[3] = ngrp;
        LM[4] = vrem;
        LM[5] = 0;
        LM[6] = act != nullptr;
        LM[7] = pbase;
        LM[8] = ngrp > 0 ? int(mlo) : 0;
        LM[9] = ngrp > 0 ? int(mhi) : 0;
        if (bad) atomicOr(a.err, 4);
      } else if (c == 1 || c == 2) {
        if (c - 1 < ngrp) M[8 + pbase + c - 1] = (j << 1) | (c - 1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.full[s]);
  }
}

// ---------------------------------------------------------------- shared pieces

struct UnitInfo {
  int unit, b, h, whole;
};

struct LoopRows {
  unsigned long long mk;  // presence of the tile's tokens
  int n, c0, g0, ngrp, pbase, vrem;
};

__device__ __forceinline__ LoopRows loop_rows(const Stage& st, int j) {
  const int32_t* LM = st.meta + 16 + kLoopMeta * j;
  const int4 la = *reinterpret_cast<const int4*>(LM);
  const int4 lb = *reinterpret_cast<const int4*>(LM + 4);
  const int2 lm = *reinterpret_cast<const int2*>(LM + 8);
  LoopRows R;
  R.n = la.x;
  R.c0 = la.y;
  R.g0 = la.z;
  R.ngrp = la.w;
  R.vrem = lb.x;
  R.pbase = lb.w;
  R.mk = (unsigned long long)uint32_t(lm.y) << 32 | uint32_t(lm.x);
  return R;
}

__device__ __forceinline__ int row_of(unsigned long long mk, int u) { return __popcll(mk & ((1ull << u) - 1ull)); }
__device__ __forceinline__ int group_of(const LoopRows& R, int row) {
  return R.ngrp > 1 ? ((R.c0 + row) >> 6) - R.g0 : 0;
}

// Bounded wait for a sequence counter to pass `target`.
__device__ __forceinline__ bool seq_wait(volatile int32_t* seq, int32_t target) {
  if (*seq > target) return true;
  const long long t0 = global_ns();
  while (*seq <= target) {
    if (global_ns() - t0 > kWaitNs) return false;
    __nanosleep(64);
  }
  return true;
}

// ---------------------------------------------------------------- softmax warps

// K-min terms q . mK of every pair into the calling warp's table (one mma.sync
// chain: rows = pairs, columns = query heads, K = channels).
template <bool G8>
__device__ void kmin_terms(Smem<G8>& S, const Stage& st, int npairs, int wq, int lane) {
  const int g = lane >> 2, q = lane & 3;
  float cc[2][4] = {};
  const bool live = g < npairs;
  const int pj = live ? st.meta[8 + g] : 0;
  const uint16_t* mrow = &st.l[pj >> 1].kmin[(pj & 1) * kD];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t a0 = live ? *reinterpret_cast<const uint32_t*>(mrow + 16 * s + 2 * q) : 0u;
    const uint32_t a2 = live ? *reinterpret_cast<const uint32_t*>(mrow + 16 * s + 2 * q + 8) : 0u;
    mma16816(cc[s & 1], a0, 0u, a2, 0u, S.qn[g][8 * s + q], S.qn[g][8 * s + q + 4]);
  }
  if (live) {
    S.kmt[wq][g][2 * q] = cc[0][0] + cc[1][0];
    S.kmt[wq][g][2 * q + 1] = cc[0][1] + cc[1][1];
  }
  __syncwarp();
}

template <int DEPTH, bool G8>
__device__ void softmax_warps(const AttnArgs& a, Smem<G8>& S, long long s0, long long e0, uint32_t tmem) {
  constexpr int kNb = Smem<G8>::kNb;
  constexpr int kSlots = G8 ? 2 : 1;
  const int tid = threadIdx.x;  // 0..127
  const int wq = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int gq = a.g;
  const float lsc = a.scale * kLog2e;
  const uint32_t tq = tmem + (uint32_t(32 * wq) << 16);
  const int ua = 16 * wq + g, uc = ua + 8;  // this thread's tokens
  float mr[kSlots], ls[kSlots], vb[2][kSlots];
#pragma unroll
  for (int e = 0; e < kSlots; ++e) {
    mr[e] = -INFINITY;
    ls[e] = 0.f;
    vb[0][e] = vb[1][e] = 0.f;
  }
  int cur_unit = -1;
  long long it = 0;
  // the unit's sums reduced over the softmax threads into slot `slot`
  auto publish_unit_sums = [&](int slot) {
#pragma unroll
    for (int e = 0; e < kSlots; ++e) {
      float l = ls[e], v0 = vb[0][e], v1 = vb[1][e];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l += __shfl_xor_sync(0xffffffffu, l, off);
        v0 += __shfl_xor_sync(0xffffffffu, v0, off);
        v1 += __shfl_xor_sync(0xffffffffu, v1, off);
      }
      const int hh = q + 4 * e;
      if (g == 0) {
        S.lsum[slot][wq][hh] = l;
        S.vbs[slot][wq][0][hh] = v0;
        S.vbs[slot][wq][1][hh] = v1;
        if (wq == 0) S.fm[slot][hh] = mr[e];
      }
    }
  };

  for (long long x = s0; x < e0; ++x, ++it) {
    const int s = int(it % kStages);
    const uint32_t tp = uint32_t(it & 1);
    const bool full_ok = mbar_wait(&S.full[s], uint32_t((it / kStages) & 1));
    if (group_sync_or(1, !full_ok || S.abort != 0)) {
      S.abort = 1;
      break;
    }
    const Stage& st = S.st[s];
    const int4 m0 = *reinterpret_cast<const int4*>(&st.meta[0]);
    const int4 m1 = *reinterpret_cast<const int4*>(&st.meta[4]);
    const int unit = m0.x, nvalid = m1.x, npairs = m1.z, tfirst = m1.w;
    if (unit != cur_unit) {
      if (cur_unit >= 0) publish_unit_sums(int(it & 1));
#pragma unroll
      for (int e = 0; e < kSlots; ++e) {
        mr[e] = -INFINITY;
        ls[e] = 0.f;
        vb[0][e] = vb[1][e] = 0.f;
      }
      cur_unit = unit;
      for (int i = tid; i < 8 * 64; i += 128) {
        const int hh = i >> 6, cc = i & 63;
        const uint16_t* qr = a.q + ((long long)m0.y * a.Hq + (long long)m0.z * gq + hh) * kD;
        S.qn[hh][cc] = hh < gq ? h2u(__floats2half2_rn(bf16_bits_to_f32(qr[2 * cc]), bf16_bits_to_f32(qr[2 * cc + 1])))
                               : 0u;
      }
      softmax_sync();
    }
    __threadfence_block();
    if (tid == 0) S.sums_seq = int32_t(it + 1);  // the unit sums of this tile's slot (if any) are in place
    kmin_terms<G8>(S, st, npairs, wq, lane);

    // ---- logits: the QK accumulators of every loop (read, then released to the next tile's QK)
    LoopRows R[DEPTH];
#pragma unroll
    for (int j = 0; j < DEPTH; ++j) R[j] = loop_rows(st, j);
    bool ok = mbar_wait(&S.mbS, tp);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) S.abort = 1;
    tc_fence_after();
    uint32_t d[DEPTH][2][kSlots][4];
#pragma unroll
    for (int j = 0; j < DEPTH; ++j)
#pragma unroll
      for (int G = 0; G < 2; ++G)
#pragma unroll
        for (int e = 0; e < kSlots; ++e) d[j][G][e][0] = d[j][G][e][1] = d[j][G][e][2] = d[j][G][e][3] = 0u;
    if (ok) {
#pragma unroll
      for (int j = 0; j < DEPTH; ++j) {
        if (R[j].ngrp == 0) continue;
#pragma unroll
        for (int e = 0; e < kSlots; ++e) {
          tmem_ld_16x256b_x1(tq + kColS + 32u * uint32_t(j) + 8u * e, d[j][0][e]);
          if (R[j].ngrp > 1) tmem_ld_16x256b_x1(tq + kColS + 32u * uint32_t(j) + uint32_t(kNb) + 8u * e, d[j][1][e]);
        }
      }
      tmem_wait_ld(d[0][0][0]);
#pragma unroll
      for (int j = 0; j < DEPTH; ++j)
#pragma unroll
        for (int G = 0; G < 2; ++G)
#pragma unroll
          for (int e = 0; e < kSlots; ++e)
            if (j + G + e > 0) tmem_touch(d[j][G][e]);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.sread);
    float sA[kSlots], sC[kSlots];
    {
      float xa[kSlots], xc[kSlots];
#pragma unroll
      for (int e = 0; e < kSlots; ++e) xa[e] = xc[e] = 0.f;
#pragma unroll
      for (int j = 0; j < DEPTH; ++j) {
        const bool pa = (R[j].mk >> ua) & 1, pc = (R[j].mk >> uc) & 1;
        const int Ga = group_of(R[j], row_of(R[j].mk, ua)), Gc = group_of(R[j], row_of(R[j].mk, uc));
#pragma unroll
        for (int e = 0; e < kSlots; ++e) {
          const int hh = q + 4 * e;
          const uint32_t* da = Ga ? d[j][1][e] : d[j][0][e];
          const uint32_t* dc = Gc ? d[j][1][e] : d[j][0][e];
          if (pa) xa[e] += (__uint_as_float(da[0]) + __uint_as_float(da[1])) * 16777216.0f + S.kmt[wq][R[j].pbase + Ga][hh];
          if (pc) xc[e] += (__uint_as_float(dc[2]) + __uint_as_float(dc[3])) * 16777216.0f + S.kmt[wq][R[j].pbase + Gc][hh];
        }
      }
      const bool vA = ok && npairs > 0 && ua < nvalid && ua >= tfirst;
      const bool vC = ok && npairs > 0 && uc < nvalid && uc >= tfirst;
#pragma unroll
      for (int e = 0; e < kSlots; ++e) {
        const bool hok = q + 4 * e < gq;
        sA[e] = (vA && hok) ? xa[e] * lsc : -INFINITY;
        sC[e] = (vC && hok) ? xc[e] * lsc : -INFINITY;
        float mt = fmaxf(sA[e], sC[e]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
        if (g == 0) S.red[wq][q + 4 * e] = mt;
      }
    }
    if (group_sync_or(1, !ok || S.abort != 0)) {  // the warps' maxima are in place
      S.abort = 1;
      break;
    }

    // ---- probabilities, P' (B of PV) and the V-min terms
    float pA[kSlots], pC[kSlots];
#pragma unroll
    for (int e = 0; e < kSlots; ++e) {
      const int hh = q + 4 * e;
      const float mg = fmaxf(fmaxf(S.red[0][hh], S.red[1][hh]), fmaxf(S.red[2][hh], S.red[3][hh]));
      const float mn = fmaxf(mr[e], mg);
      const float al = (mr[e] == -INFINITY) ? 0.f : exp2f(mr[e] - mn);
      mr[e] = mn;
      pA[e] = sA[e] == -INFINITY ? 0.f : exp2f(sA[e] - mn);
      pC[e] = sC[e] == -INFINITY ? 0.f : exp2f(sC[e] - mn);
      ls[e] = ls[e] * al + (pA[e] + pC[e]);
      vb[0][e] *= al;
      vb[1][e] *= al;
      if (wq == 0 && g == 0) S.alpha[tp][hh] = al;
    }
    uint8_t* bpt = reinterpret_cast<uint8_t*>(S.bp[tp]);
#pragma unroll
    for (int j = 0; j < DEPTH; ++j) {
      const bool pa = (R[j].mk >> ua) & 1, pc = (R[j].mk >> uc) & 1;
      const int ra = row_of(R[j].mk, ua), rc = row_of(R[j].mk, uc);
      float2 sva = make_float2(0.f, 0.f), svc = sva, mva = sva, mvc = sva;
      if (pa) {
        sva = __half22float2(u2h(*reinterpret_cast<const uint32_t*>(&st.l[j].vsc[R[j].vrem + 2 * ra])));
        mva = __half22float2(u2h(*reinterpret_cast<const uint32_t*>(&st.l[j].vmin[R[j].vrem + 2 * ra])));
      }
      if (pc) {
        svc = __half22float2(u2h(*reinterpret_cast<const uint32_t*>(&st.l[j].vsc[R[j].vrem + 2 * rc])));
        mvc = __half22float2(u2h(*reinterpret_cast<const uint32_t*>(&st.l[j].vmin[R[j].vrem + 2 * rc])));
      }
      uint8_t* bpj = bpt + j * (KVQ_TILE * 16 * 2);
#pragma unroll
      for (int e = 0; e < kSlots; ++e) {
        const int hh = q + 4 * e;
        if (hh >= gq) continue;
        const float qa = pa ? pA[e] : 0.f, qc = pc ? pC[e] : 0.f;
        const int nb = ((2 * hh) >> 3) * 1024 + ((2 * hh) & 7) * 2;
        *reinterpret_cast<uint32_t*>(bpj + nb + (ua >> 3) * 128 + (ua & 7) * 16) =
            h2u(__floats2half2_rn(qa * sva.x, qa * sva.y));
        *reinterpret_cast<uint32_t*>(bpj + nb + (uc >> 3) * 128 + (uc & 7) * 16) =
            h2u(__floats2half2_rn(qc * svc.x, qc * svc.y));
        vb[0][e] = fmaf(qa, mva.x, fmaf(qc, mvc.x, vb[0][e]));
        vb[1][e] = fmaf(qa, mva.y, fmaf(qc, mvc.y, vb[1][e]));
      }
    }
    fence_async_smem();
    // the PV issuers have taken the previous P' (keeps this barrier within one phase of its waiters)
    if (it > 0 && !__all_sync(0xffffffffu, mbar_wait(&S.mbO, tp ^ 1u))) S.abort = 1;
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&S.pready);
      mbar_arrive(&S.empty[s]);
    }
    __threadfence_block();
    if (tid == 0) S.alpha_seq = int32_t(it + 1);
  }
  // the last unit's sums
  if (!S.abort && it > 0) publish_unit_sums(int(it & 1));
  __threadfence_block();
  softmax_sync();
  if (tid == 0) S.sums_seq = int32_t(it + 1);
}

// ---------------------------------------------------------------- operand warps

template <int DEPTH, bool G8>
__device__ void operand_warps(const AttnArgs& a, Smem<G8>& S, int vcta, long long s0, long long e0, uint32_t tmem) {
  constexpr int kNb = Smem<G8>::kNb;
  const int ot = threadIdx.x - 32 * kWarpOperand;  // 0..127
  const int wq = ot >> 5, lane = ot & 31;
  const int g = lane >> 2, q = lane & 3;
  const int gq = a.g;
  const uint32_t tq = tmem + (uint32_t(32 * wq) << 16);
  // fold state: channel row m of the PV accumulators
  const int m_row = ot;
  const int ch_m = 32 * (m_row >> 5) + 8 * ((m_row >> 3) & 3) + ((m_row & 7) >> 1) + 4 * (m_row & 1);
  const int vg_m = m_row >> 6;
  const float rs_m = (((m_row & 7) >> 1) & 1) ? 1048576.0f : 16777216.0f;  // odd-e rows carry 2^-20
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const uint32_t idPV = instr_desc(128, 16, 1, 1);
  (void)idPV;
  int q_unit = -1;
  UnitInfo cu = {-1, 0, 0, 0}, pu = {-1, 0, 0, 0};
  long long it = 0;

  // Output of a finished unit (its sums in slot `slot`): acc with the row
  // scale plus the V-min terms, over the sum, or the unnormalised partial slot.
  auto finish_unit = [&](const UnitInfo& U, int slot) {
    float* ps = a.partials + (size_t)(blockIdx.x + U.unit) * kSlotFloats;
    for (int hh = 0; hh < gq; ++hh) {
      const float lt = S.lsum[slot][0][hh] + S.lsum[slot][1][hh] + S.lsum[slot][2][hh] + S.lsum[slot][3][hh];
      const float vbt = S.vbs[slot][0][vg_m][hh] + S.vbs[slot][1][vg_m][hh] + S.vbs[slot][2][vg_m][hh] +
                        S.vbs[slot][3][vg_m][hh];
      float av = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) av = (i == hh) ? acc[i] : av;
      const float o = av * rs_m + vbt;
      const long long qrow = (long long)U.b * a.Hq + (long long)U.h * gq + hh;
      if (U.whole) {
        a.out[qrow * kD + ch_m] = o / lt;
        if (m_row == 0) a.stats[qrow] = make_float2(S.fm[slot][hh], lt);
      } else {
        ps[2 * kMaxG + hh * kD + ch_m] = o;
        if (m_row == 0) {
          ps[kMaxG + hh] = lt;
          ps[hh] = S.fm[slot][hh];
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  };
  // fold of the PV accumulators of tile `t` (complete) with that tile's rescale
  auto fold = [&](long long t) {
    uint32_t v[16], v2[16];
    tmem_ld_32x32b_x16(tq + kColO, v);
    if (DEPTH > 1) tmem_ld_32x32b_x16(tq + kColO + 16, v2);
    const float* al = S.alpha[t & 1];
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) {
      if (hh < gq) {
        float dd = __uint_as_float(vg_m ? v[2 * hh + 1] : v[2 * hh]);
        if (DEPTH > 1) dd += __uint_as_float(vg_m ? v2[2 * hh + 1] : v2[2 * hh]);
        acc[hh] = acc[hh] * al[hh] + dd;
      }
    }
  };

  bool ok = true;
  for (long long x = s0; x < e0; ++x, ++it) {
    const int s = int(it % kStages);
    const bool full_ok = mbar_wait(&S.full[s], uint32_t((it / kStages) & 1));
    if (group_sync_or(2, !full_ok || S.abort != 0)) {
      S.abort = 1;
      break;
    }
    const Stage& st = S.st[s];
    const int4 m0 = *reinterpret_cast<const int4*>(&st.meta[0]);
    const int4 m1 = *reinterpret_cast<const int4*>(&st.meta[4]);
    cu.unit = m0.x;
    cu.b = m0.y;
    cu.h = m0.z;
    cu.whole = m1.y;
    if (cu.unit != q_unit) {  // the unit's q in QK k order (every operand thread is past the previous tile's use)
      for (int i = ot; i < 8 * 64; i += 128) {
        const int hh = i >> 6, c = i & 63;
        const uint16_t* qr = a.q + ((long long)cu.b * a.Hq + (long long)cu.h * gq + hh) * kD;
        const int kb = c >> 2, m = c & 3;
        const int ch = 32 * m + 8 * (kb >> 2) + (kb & 3);
        const float f = (kb & 1) ? 0.0625f : 1.0f;
        S.qp[hh][c] = hh < gq ? h2u(__floats2half2_rn(bf16_bits_to_f32(qr[ch]) * f, bf16_bits_to_f32(qr[ch + 4]) * f))
                              : 0u;
      }
      q_unit = cu.unit;
      operand_sync();
    }
    LoopRows R[DEPTH];
#pragma unroll
    for (int j = 0; j < DEPTH; ++j) R[j] = loop_rows(st, j);
    // the previous tile's QK has read the operands
    if (it > 0) ok = __all_sync(0xffffffffu, mbar_wait(&S.mbS, uint32_t((it - 1) & 1)));
    if (!ok) {  // the next tile's group check ends the loop
      S.abort = 1;
      continue;
    }
    tc_fence_after();

    // ---- Q' (B of QK): item (loop, K group, head, k block)
#pragma unroll
    for (int j = 0; j < DEPTH; ++j) {
      const int per_group = gq * 16;
      const int items = R[j].ngrp * per_group;
      for (int i2 = ot; i2 < items; i2 += 128) {
        const int G = i2 / per_group, r = i2 % per_group;
        const int hh = r >> 4, kb = r & 15;
        const uint16_t* sc = &st.l[j].ksc[G * kD];
        const int cb = 8 * (kb >> 2) + (kb & 3);
        uint32_t sp[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) sp[m] = uint32_t(sc[cb + 32 * m]) | (uint32_t(sc[cb + 32 * m + 4]) << 16);
        const uint4 qv = *reinterpret_cast<const uint4*>(&S.qp[hh][4 * kb]);
        const uint32_t qa[4] = {qv.x, qv.y, qv.z, qv.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const __half2 hv = __hmul2(u2h(qa[m]), u2h(sp[m]));  // RN16(q * s)
          hi[m] = h2u(hv);
          lo[m] = h2u(__hfma2(u2h(qa[m]), u2h(sp[m]), __hneg2(hv)));  // RN16(q * s - hi)
        }
        const int n = G * kNb + 2 * hh;
        uint8_t* row =
            reinterpret_cast<uint8_t*>(S.bq + Smem<G8>::bq_off(j)) + (n >> 3) * 2048 + kb * 128 + (n & 7) * 16;
        *reinterpret_cast<uint4*>(row) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(row + 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    // ---- K codes (A of QK) into tensor memory: thread (g, q) takes chunk q of tokens 16 wq + g, + 8
    {
      const int ua = 16 * wq + g, uc = ua + 8;
      uint4 wa[DEPTH], wb[DEPTH];
#pragma unroll
      for (int j = 0; j < DEPTH; ++j) {
        const bool pa = R[j].ngrp > 0 && ((R[j].mk >> ua) & 1), pc = R[j].ngrp > 0 && ((R[j].mk >> uc) & 1);
        wa[j] = pa ? *reinterpret_cast<const uint4*>(&st.l[j].kc[row_of(R[j].mk, ua) * kRowBytes + 16 * q])
                   : make_uint4(0, 0, 0, 0);
        wb[j] = pc ? *reinterpret_cast<const uint4*>(&st.l[j].kc[row_of(R[j].mk, uc) * kRowBytes + 16 * q])
                   : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < DEPTH; ++j) {
        if (R[j].ngrp == 0) continue;
        const uint32_t wA[4] = {wa[j].x, wa[j].y, wa[j].z, wa[j].w}, wB[4] = {wb[j].x, wb[j].y, wb[j].z, wb[j].w};
#pragma unroll
        for (int hw = 0; hw < 2; ++hw) {
          uint32_t r[16];
#pragma unroll
          for (int i2 = 0; i2 < 2; ++i2) {
            const int i = 2 * hw + i2;
            const uint32_t xa = wA[i], xb = wB[i], ya = xa >> 8, yb = xb >> 8;
            r[8 * i2 + 0] = xa & kLoMask;
            r[8 * i2 + 1] = xb & kLoMask;
            r[8 * i2 + 2] = xa & kHiMask;
            r[8 * i2 + 3] = xb & kHiMask;
            r[8 * i2 + 4] = ya & kLoMask;
            r[8 * i2 + 5] = yb & kLoMask;
            r[8 * i2 + 6] = ya & kHiMask;
            r[8 * i2 + 7] = yb & kHiMask;
          }
          tmem_st_16x128b_x8(tq + kColA + 64u * uint32_t(j) + 32u * hw, r);
        }
      }
    }
    tmem_wait_st();
    fence_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.ops);

    // ---- the previous tile's PV: fold, and the output of a unit that ended with it
    if (it > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&S.mbO, uint32_t((it - 1) & 1)) && seq_wait(&S.alpha_seq, int32_t(it - 1)));
      if (!ok) {
        S.abort = 1;
        continue;
      }
      __threadfence_block();
      tc_fence_after();
      fold(it - 1);
      if (pu.unit != cu.unit) {
        ok = __all_sync(0xffffffffu, seq_wait(&S.sums_seq, int32_t(it)));
        if (!ok) {
          S.abort = 1;
          continue;
        }
        __threadfence_block();
        finish_unit(pu, int(it & 1));
      }
    }
    // ---- V codes (A of PV) into shared memory: thread (token u, half hv), rotated chunks
    {
      const int hv = wq >> 1, u = 32 * (wq & 1) + lane;
#pragma unroll
      for (int j = 0; j < DEPTH; ++j) {
        if (R[j].ngrp == 0 || !((R[j].mk >> u) & 1)) continue;
        const int rr = row_of(R[j].mk, u);
        uint8_t* vdst = reinterpret_cast<uint8_t*>(S.va[j]) + (u >> 3) * 128 + (u & 7) * 16;
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          const int cch = (2 * hv + s2 + ((lane >> 1) & 3)) & 3;  // conflict-free loads
          const uint4 x4 = *reinterpret_cast<const uint4*>(&st.l[j].vc[rr * kRowBytes + 16 * cch]);
          const uint32_t X[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t xx = X[i], yy = xx >> 8;
            *reinterpret_cast<uint4*>(vdst + (4 * cch + i) * 1024) =
                make_uint4(xx & kLoMask, xx & kHiMask, yy & kLoMask, yy & kHiMask);
          }
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&S.vready);
      mbar_arrive(&S.empty[s]);
    }
    pu = cu;
  }
  // ---- drain: the last tile's PV, its fold and the unit's output
  if (!S.abort && it > 0) {
    ok = __all_sync(0xffffffffu, mbar_wait(&S.mbO, uint32_t((it - 1) & 1)) && seq_wait(&S.alpha_seq, int32_t(it - 1)) &&
                                     seq_wait(&S.sums_seq, int32_t(it)));
    if (ok) {
      __threadfence_block();
      tc_fence_after();
      fold(it - 1);
      finish_unit(pu, int(it & 1));
    } else {
      S.abort = 1;
    }
  }
  (void)vcta;
}

// ---------------------------------------------------------------- MMA issuers
//
// One thread of warp 8 + j: per tile, the QK MMAs of loop j once the operands
// are written and the previous tile's accumulators read (a commit to mbS in any
// case, so that mbS completes once per tile). One thread of warp 12 + p: the PV
// MMAs of loops p, p + 2 once P' and the V operands are written. The stage's
// metadata stays valid until the softmax warps release the stage, after mbS.
template <int DEPTH, bool G8>
__device__ void qk_issuer(const AttnArgs& a, Smem<G8>& S, int j, long long s0, long long e0, uint32_t tmem) {
  constexpr int kNb = Smem<G8>::kNb;
  const uint64_t bq_desc = smem_desc(smem_addr(S.bq + Smem<G8>::bq_off(j)), 128, 2048);
  long long it = 0;
  for (long long x = s0; x < e0 && !S.abort; ++x, ++it) {
    if (!mbar_wait(&S.ops, uint32_t(it & 1)) || (it > 0 && !mbar_wait(&S.sread, uint32_t((it - 1) & 1)))) {
      S.abort = 1;
      atomicOr(a.err, 8);
      break;
    }
    tc_fence_after();
    const int ngrp = S.st[int(it % kStages)].meta[16 + kLoopMeta * j + 3];
    if (ngrp > 0) {
      const uint32_t idQK = instr_desc(64, ngrp * kNb, 0, 0);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_ts(tmem + kColS + 32u * uint32_t(j), tmem + kColA + 64u * uint32_t(j) + 8u * k, bq_desc + 16ull * k, idQK,
               k != 0);
    }
    mma_commit(&S.mbS);
  }
}

template <int DEPTH, bool G8>
__device__ void pv_issuer(const AttnArgs& a, Smem<G8>& S, int p, long long s0, long long e0, uint32_t tmem) {
  const uint32_t idPV = instr_desc(128, 16, 1, 1);
  long long it = 0;
  for (long long x = s0; x < e0 && !S.abort; ++x, ++it) {
    const uint32_t tp = uint32_t(it & 1);
    if (!mbar_wait(&S.pready, tp) || !mbar_wait(&S.vready, tp)) {
      S.abort = 1;
      atomicOr(a.err, 8);
      break;
    }
    tc_fence_after();
#pragma unroll
    for (int jj = p; jj < DEPTH; jj += 2) {
      const uint64_t ad = smem_desc(smem_addr(S.va[jj]), 128, 1024);
      const uint64_t bd = smem_desc(smem_addr(S.bp[tp][jj]), 128, 1024);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_ss(tmem + kColO + 16u * uint32_t(p), ad + 16ull * k, bd + 16ull * k, idPV, (jj != p) || (k != 0));
    }
    mma_commit(&S.mbO);
  }
}

template <int DEPTH, bool G8>
__global__ void __launch_bounds__(kThreads, 1) attn_tcgen05_kernel(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<G8>& S = *reinterpret_cast<Smem<G8>*>(smem_raw);
  constexpr int kPvIssuers = DEPTH < 2 ? DEPTH : 2;
  constexpr int kIssuers = DEPTH + kPvIssuers;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], 8);
    }
    mbar_init(&S.ops, 4);
    mbar_init(&S.sread, 4);
    mbar_init(&S.pready, 4);
    mbar_init(&S.vready, 4);
    mbar_init(&S.mbS, DEPTH);
    mbar_init(&S.mbO, kPvIssuers);
    mbar_init(&S.drain, kIssuers);
    S.abort = 0;
    S.alpha_seq = 0;
    S.sums_seq = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // operand areas start zeroed: B columns of absent query heads stay zero, and
  // the V operand rows of tokens a loop does not store hold finite values
  {
    uint4* z = reinterpret_cast<uint4*>(&S);
    const int n16 = int((sizeof(S.va) + sizeof(S.bq) + sizeof(S.bp)) / 16);
    for (int i = threadIdx.x; i < n16; i += kThreads) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  wait_prior_grid();  // the plan (tile prefix, error word) is complete and visible from here on
  const long long W = a.prefix[a.n_requests];
  const int C = a.n_ctas;
  const long long s0 = cta_start(blockIdx.x, W, C), e0 = cta_start(blockIdx.x + 1, W, C);
  if (s0 >= e0) return;
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&S.tmem)),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kWarpProducer) {
    producer<DEPTH, G8>(a, S, warp - kWarpProducer, s0, e0, lane);
    return;
  }
  if (warp < kWarpOperand) {
    softmax_warps<DEPTH, G8>(a, S, s0, e0, tmem);
  } else if (warp < kWarpQk) {
    operand_warps<DEPTH, G8>(a, S, blockIdx.x, s0, e0, tmem);
  } else {
    const bool qk = warp < kWarpPv;
    const int idx = qk ? warp - kWarpQk : warp - kWarpPv;
    const bool active = qk ? idx < DEPTH : idx < kPvIssuers;
    if (active && lane == 0) {
      if (qk) qk_issuer<DEPTH, G8>(a, S, idx, s0, e0, tmem);
      else pv_issuer<DEPTH, G8>(a, S, idx, s0, e0, tmem);
      // every MMA this thread issued is complete before the tensor memory is freed
      mma_commit(&S.drain);
      (void)mbar_wait(&S.drain, 0u);
    }
    __syncwarp();
  }
  if (S.abort && threadIdx.x == 0) atomicOr(a.err, 8);
  tc_fence_before();
  tmem_users_sync();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
  }
}

template <int DEPTH, bool G8>
cudaError_t launch_depth(const AttnArgs& a, cudaStream_t stream) {
  const int smem = int(sizeof(Smem<G8>));
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_tcgen05_kernel<DEPTH, G8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_dependent(attn_tcgen05_kernel<DEPTH, G8>, dim3(a.n_ctas), dim3(kThreads), size_t(smem), stream, a);
}

static_assert(sizeof(Smem<true>) <= 227 * 1024, "one block per SM: at most 227 KB of shared memory");

}  // namespace t5_attn

// The INT4 packed attention on tcgen05 (dense calls, depth <= 4, 1/2/4/8 query
// heads per KV head); one block per SM, one CTA of the work split per block.
cudaError_t launch_attn_tcgen05(const AttnArgs& a, cudaStream_t stream) {
  using namespace t5_attn;
  cudaError_t e;
  switch (a.depth * 2 + (a.g == 8 ? 1 : 0)) {
    case 2: e = launch_depth<1, false>(a, stream); break;
    case 3: e = launch_depth<1, true>(a, stream); break;
    case 4: e = launch_depth<2, false>(a, stream); break;
    case 5: e = launch_depth<2, true>(a, stream); break;
    case 6: e = launch_depth<3, false>(a, stream); break;
    case 7: e = launch_depth<3, true>(a, stream); break;
    case 8: e = launch_depth<4, false>(a, stream); break;
    case 9: e = launch_depth<4, true>(a, stream); break;
    default: return cudaErrorInvalidValue;
  }
  count_launch();
  return e;
}

}  // namespace kvq
