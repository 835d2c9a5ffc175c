// kvq_internal.cuh — device helpers shared by the codec, reconstruction and
// attention kernels of libkvq. Codec arithmetic follows the quantiser and the
// residual chain of the FlashLoop RFC (vllm-rlt issue #156) §3.3 with the FP32
// codes / FP16 metadata order of the INT4 codec PR (vllm-rlt pull #166, review
// by 0z5a). Every rounding step is an explicit round-to-nearest intrinsic, so
// FMA contraction cannot change a codec result.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kvq.h"

namespace kvq {

constexpr int kD = 128;       // head_dim supported by the kernels
constexpr int kG = KVQ_GROUP;  // 64
constexpr int kRowBytes = kD / 2;  // packed bytes per (row, head)

// Per-loop plane pointers as the kernels see them (a trimmed kvq_stream).
struct LoopPlanes {
  int32_t n_rows;
  int32_t sparse;
  int32_t ktile;    // K groups by 64-token logical tile (KVQ_KGROUP_TILE) instead of 64 stored rows
  int32_t kgroups;  // K groups per head of the param planes: ceil(n_tokens/64) if ktile, else ceil(n_rows/64),
                    // or the capacity's
  int32_t fmt;      // KVQ_FMT_INT4 or KVQ_FMT_NVFP4
  int32_t stride;   // rows per head of the planes (the row capacity; n_rows unless the stream can grow)
  const int32_t* active;
  const int32_t* tile_dir;
  const uint8_t* codes;
  const uint16_t* mins;    // INT4 (NVFP4: the E4M3 block scales, as bytes)
  const uint16_t* scales;  // INT4 (NVFP4: the tensor-scale record, as floats)
};

struct Chain {
  int32_t depth;
  int32_t kind;
  int32_t n_tokens;
  int32_t n_heads;
  int32_t any_nvfp4;  // some loop of the chain is NVFP4 (the INT4-only kernels refuse it)
  int32_t pad[3];
  LoopPlanes loop[KVQ_MAX_LOOPS];
};

// ---- NVFP4 element and scale types, written from the format definitions
// (codec PR review by 0z5a: E2M1 round-to-nearest-even, E4M3 scale rounding).

// E4M3 (finite variant: bias 7, subnormals m * 2^-9, largest 448) to FP32.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t E = (b >> 3) & 15u, M = b & 7u;
  const float mag = E ? __uint_as_float(((E + 120u) << 23) | (M << 20)) : float(M) * 0.001953125f;
  return (b & 0x80u) ? -mag : mag;
}

// E4M3 byte of v >= 0: round to nearest even (three mantissa bits), saturating at 448.
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  if (!(v < 448.0f)) return 0x7Eu;
  if (v < 0.015625f) {  // below 2^-6: a multiple of 2^-9 (v * 512 < 8 is exact; adding 2^23 rounds it)
    const float m = __fsub_rn(__fadd_rn(__fmul_rn(v, 512.0f), 8388608.0f), 8388608.0f);
    return m >= 8.0f ? 0x08u : uint32_t(m);
  }
  uint32_t u = __float_as_uint(v);
  u += 0x7FFFFu + ((u >> 20) & 1u);  // ties to even at the third mantissa bit; a carry bumps the exponent
  u &= 0xFFF00000u;
  return (((u >> 23) - 120u) << 3) | ((u >> 20) & 7u);
}

// E2M1 nibble (sign in bit 3; magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6) to FP32.
__device__ __forceinline__ float e2m1_to_f32(uint32_t n) {
  const uint32_t c = n & 7u;
  const float mag = c >= 2u ? __uint_as_float((((c >> 1) + 126u) << 23) | ((c & 1u) << 22)) : 0.5f * float(c);
  return (n & 8u) ? -mag : mag;
}

// E2M1 nibble of y: the nearest magnitude (ties to the even code, i.e. to the
// even mantissa), saturating at 6, with the sign bit of y.
__device__ __forceinline__ uint32_t f32_to_e2m1(float y) {
  const float a = fabsf(y);
  const uint32_t c = uint32_t(a > 0.25f) + uint32_t(a >= 0.75f) + uint32_t(a > 1.25f) + uint32_t(a >= 1.75f) +
                     uint32_t(a > 2.5f) + uint32_t(a >= 3.5f) + uint32_t(a > 5.0f);
  return c | ((__float_as_uint(y) >> 28) & 8u);
}

// One NVFP4 element in FP32: RN32(RN32(e2m1 * s_b) * s_t), the inner product exact.
__device__ __forceinline__ float nvfp4_dequant(uint32_t nib, float sb, float st) {
  return __fmul_rn(__fmul_rn(e2m1_to_f32(nib), sb), st);
}

// Two E2M1 codes (the low byte of x: low nibble, high nibble) as an exact FP16
// pair {low, high}, by the hardware conversion.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t x) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(r) : "r"(x));
  return r;
}

// Two E4M3 values (the low 16 bits of x) as an exact FP16 pair {low byte, high byte}.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t x) {
  uint32_t r;
  asm("{\n\t.reg .b16 h;\n\tcvt.u16.u32 h, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(r) : "r"(x));
  return r;
}

// NVFP4 planes of a loop: E4M3 block scale of (head h, stored row, block of 16
// channels) and the tensor scale.
__device__ __forceinline__ float nvfp4_block_scale(const LoopPlanes& L, int h, int row, int blk) {
  return e4m3_to_f32(__ldg(reinterpret_cast<const uint8_t*>(L.mins) + ((long long)h * L.stride + row) * (kD / 16) + blk));
}
__device__ __forceinline__ float nvfp4_tensor_scale(const LoopPlanes& L) {
  return __ldg(reinterpret_cast<const float*>(L.scales));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float round_bf16(float f) { return bf16_bits_to_f32(f32_to_bf16_bits(f)); }
__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ uint16_t f32_to_f16_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }

// decode(c) = RN_bf16(RN32(min16 + RN32(scale16 * c))).
__device__ __forceinline__ float dequant(uint16_t min16, uint16_t scale16, int c) {
  return round_bf16(__fadd_rn(f16_bits_to_f32(min16), __fmul_rn(f16_bits_to_f32(scale16), float(c))));
}

// Compact row of logical token t in a sparse loop, or -1 if t is absent. The
// tile directory narrows the search to the <= 64 indices of t's 64-token tile.
__device__ __forceinline__ int sparse_rank(const LoopPlanes& L, int t) {
  int lo = __ldg(L.tile_dir + (t >> 6));
  int hi = __ldg(L.tile_dir + (t >> 6) + 1);
  if (lo < 0) lo = 0;
  if (hi > L.n_rows) hi = L.n_rows;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    int v = __ldg(L.active + mid);
    if (v < t) lo = mid + 1;
    else hi = mid;
  }
  if (lo < L.n_rows && lo < __ldg(L.tile_dir + (t >> 6) + 1) && __ldg(L.active + lo) == t) return lo;
  return -1;
}

__device__ __forceinline__ int row_of(const LoopPlanes& L, int t) { return L.sparse ? sparse_rank(L, t) : t; }

// K groups per head of a loop with n_rows stored rows of n_tokens tokens.
__host__ __device__ __forceinline__ int k_groups_of(bool ktile, int n_rows, int n_tokens) {
  if (n_rows <= 0) return 0;
  return ktile ? (n_tokens + kG - 1) / kG : (n_rows + kG - 1) / kG;
}

// K group of the stored row `row` of logical token t: its 64-token logical tile
// under tile grouping, else its block of 64 stored rows (the same for a dense loop).
__device__ __forceinline__ int k_group(const LoopPlanes& L, int t, int row) { return L.ktile ? (t >> 6) : (row >> 6); }

// Index of the params of (head h, logical token t stored at `row`, channel d).
__device__ __forceinline__ long long param_index(int kind, const LoopPlanes& L, int h, int t, int row, int d) {
  if (kind == KVQ_K) return ((long long)h * L.kgroups + k_group(L, t, row)) * kD + d;
  return ((long long)h * L.stride + row) * (kD / kG) + d / kG;
}

// Loop j of request R as the K (kind 0) or V planes the kernels read.
__device__ __forceinline__ void planes_of(const kvq_request& R, int j, int kind, LoopPlanes& P) {
  const kvq_loop_ref& L = R.loop[j];
  P.n_rows = L.n_rows;
  P.sparse = L.active_idx != nullptr;
  P.ktile = kind == KVQ_K && (L.flags & KVQ_LOOP_K_TILE) != 0;
  P.kgroups = L.kgroup_cap > 0 ? L.kgroup_cap : k_groups_of(P.ktile != 0, L.n_rows, R.n_tokens);
  P.stride = L.row_cap > 0 ? L.row_cap : L.n_rows;
  P.fmt = (L.flags & (kind == KVQ_K ? KVQ_LOOP_K_NVFP4 : KVQ_LOOP_V_NVFP4)) ? KVQ_FMT_NVFP4 : KVQ_FMT_INT4;
  P.active = L.active_idx;
  P.tile_dir = L.tile_dir;
  P.codes = kind == KVQ_K ? L.k_codes : L.v_codes;
  P.mins = kind == KVQ_K ? L.k_mins : L.v_mins;
  P.scales = kind == KVQ_K ? L.k_scales : L.v_scales;
}

// Reconstruct 4 consecutive channels c0..c0+3 (c0 % 4 == 0) of token t, head h,
// through loops 0..depth-1, given each loop's stored row (rows[j] < 0: absent).
__device__ __forceinline__ void chain4(const Chain& C, int depth, const int* rows, int t, int h, int c0,
                                       float out[4]) {
  {
    const LoopPlanes& B = C.loop[0];
    int row = rows[0];
    uint16_t two = *reinterpret_cast<const uint16_t*>(B.codes + ((long long)h * B.stride + row) * kRowBytes + c0 / 2);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int c = (two >> (4 * e)) & 0xF;
      long long pi = param_index(C.kind, B, h, t, row, c0 + e);
      out[e] = dequant(__ldg(B.mins + pi), __ldg(B.scales + pi), c);
    }
  }
  for (int j = 1; j < depth; ++j) {
    int row = rows[j];
    if (row < 0) continue;  // absent: inherit the predecessor
    const LoopPlanes& L = C.loop[j];
    uint16_t two = *reinterpret_cast<const uint16_t*>(L.codes + ((long long)h * L.stride + row) * kRowBytes + c0 / 2);
    if (L.fmt == KVQ_FMT_NVFP4) {  // the four channels share one 16-channel block
      const float sb = nvfp4_block_scale(L, h, row, c0 / 16), st = nvfp4_tensor_scale(L);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        out[e] = round_bf16(__fadd_rn(out[e], round_bf16(nvfp4_dequant((two >> (4 * e)) & 0xF, sb, st))));
      continue;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int c = (two >> (4 * e)) & 0xF;
      long long pi = param_index(C.kind, L, h, t, row, c0 + e);
      out[e] = round_bf16(__fadd_rn(out[e], dequant(__ldg(L.mins + pi), __ldg(L.scales + pi), c)));
    }
  }
}

// The same chain in FP32: decode = RN32(min16 + RN32(scale16 * c)), loops
// summed with FP32 rounding only (the values a direct packed reader uses).
// The four channels share one V group, and their K parameters are adjacent,
// so each loop's parameters come in one load per plane.
__device__ __forceinline__ void chain4_f32(const Chain& C, int depth, const int* rows, int t, int h, int c0,
                                           float out[4]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) out[e] = 0.0f;
  for (int j = 0; j < depth; ++j) {
    int row = rows[j];
    if (row < 0) continue;
    const LoopPlanes& L = C.loop[j];
    uint16_t two = *reinterpret_cast<const uint16_t*>(L.codes + ((long long)h * L.stride + row) * kRowBytes + c0 / 2);
    if (L.fmt == KVQ_FMT_NVFP4) {
      const float sb = nvfp4_block_scale(L, h, row, c0 / 16), st = nvfp4_tensor_scale(L);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float dq = nvfp4_dequant((two >> (4 * e)) & 0xF, sb, st);
        out[e] = (j == 0) ? dq : __fadd_rn(out[e], dq);
      }
      continue;
    }
    float mn[4], sc[4];
    if (C.kind == KVQ_K) {
      const long long pi = param_index(KVQ_K, L, h, t, row, c0);
      const uint2 m4 = __ldg(reinterpret_cast<const uint2*>(L.mins + pi));
      const uint2 s4 = __ldg(reinterpret_cast<const uint2*>(L.scales + pi));
      const uint32_t mw[2] = {m4.x, m4.y}, sw[2] = {s4.x, s4.y};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        mn[e] = f16_bits_to_f32(uint16_t(mw[e >> 1] >> (16 * (e & 1))));
        sc[e] = f16_bits_to_f32(uint16_t(sw[e >> 1] >> (16 * (e & 1))));
      }
    } else {
      const long long pi = param_index(KVQ_V, L, h, t, row, c0);
      const float m1 = f16_bits_to_f32(__ldg(L.mins + pi)), s1 = f16_bits_to_f32(__ldg(L.scales + pi));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        mn[e] = m1;
        sc[e] = s1;
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int c = (two >> (4 * e)) & 0xF;
      float dq = __fadd_rn(mn[e], __fmul_rn(sc[e], float(c)));
      out[e] = (j == 0) ? dq : __fadd_rn(out[e], dq);
    }
  }
}

// Same for one channel d.
__device__ __forceinline__ float chain1(const Chain& C, int depth, const int* rows, int t, int h, int d) {
  float v;
  {
    const LoopPlanes& B = C.loop[0];
    int row = rows[0];
    uint8_t byte = __ldg(B.codes + ((long long)h * B.stride + row) * kRowBytes + d / 2);
    int c = (d & 1) ? (byte >> 4) : (byte & 0xF);
    long long pi = param_index(C.kind, B, h, t, row, d);
    v = dequant(__ldg(B.mins + pi), __ldg(B.scales + pi), c);
  }
  for (int j = 1; j < depth; ++j) {
    int row = rows[j];
    if (row < 0) continue;
    const LoopPlanes& L = C.loop[j];
    uint8_t byte = __ldg(L.codes + ((long long)h * L.stride + row) * kRowBytes + d / 2);
    int c = (d & 1) ? (byte >> 4) : (byte & 0xF);
    if (L.fmt == KVQ_FMT_NVFP4) {
      v = round_bf16(__fadd_rn(v, round_bf16(nvfp4_dequant(c, nvfp4_block_scale(L, h, row, d / 16),
                                                           nvfp4_tensor_scale(L)))));
      continue;
    }
    long long pi = param_index(C.kind, L, h, t, row, d);
    v = round_bf16(__fadd_rn(v, dequant(__ldg(L.mins + pi), __ldg(L.scales + pi), c)));
  }
  return v;
}

// Number of kernels this library has launched in the process (host counter).
void count_launch();

enum { kModeEncK = 0, kModeEncV = 1, kModeTileDir = 2, kModeRecon = 3, kModeReconK = 4, kModeNvAmax = 5,
       kModeNvEnc = 6 };

// Arguments of the codec kernels: either a batch described by a device table of
// requests, or one request carried by value in the kernel parameters.
struct CodecArgs {
  const kvq_request* reqs;   // device table [n_requests], or nullptr: use `one`
  const uint16_t* const* x;  // batch encode: device array of BF16 [T_b][H][D] sources
  uint16_t* const* out;      // batch reconstruct: device array of BF16 [T_b][H][D] outputs
  int32_t* err;              // error word, or nullptr
  int32_t n_requests;
  int32_t H;
  int32_t kind;
  int32_t loop;              // encode and tile directory: loop written; reconstruct: depth
  uint32_t nvfp4;            // bit j: loop j of `kind` is NVFP4 in every request
  int32_t append;            // batch encode of the last 64-token tile only (the table already counts it)
  const int32_t* skip;       // append: requests to leave alone (device [n_requests]), or nullptr
  kvq_request one;
  const uint16_t* one_x;
  uint16_t* one_out;
  int32_t one_prefix[2];
};

// Index extension of a tile append (kvq_append_tile): per sparse loop, the
// tile's relative positions (checked into `rel_ws`), their absolute indices
// after the n_old stored rows, the tile directory entries of the new tile, and
// a two-entry directory of the tile alone for the encode of its rows.
struct AppendIndexArgs {
  int32_t n_loops;
  int32_t T;        // tokens before the tile (a multiple of 64)
  int32_t* err;
  struct Loop {
    const int32_t* rel;  // caller's positions 0..63 (NULL: dense loop)
    int32_t* rel_ws;     // [64] checked copy
    int32_t* dir_ws;     // [2] = {0, n_new}
    int32_t* active;     // the stream's index plane
    int32_t* tile_dir;   // the stream's tile directory
    int32_t n_old, n_new;
  } loop[KVQ_MAX_LOOPS];
};
cudaError_t launch_append_index(const AppendIndexArgs& a, cudaStream_t stream);

// Batched tile append (kvq_append_tile_batch): checks, index extension and the
// table update for every request of a device table, before the encodes.
struct AppendBatchArgs {
  kvq_request* reqs;
  int32_t n_requests;
  int32_t n_loops;
  int32_t H;
  const int32_t* const* tile_active;  // [n_loops * n_requests], loop-major; NULL entries: dense loops
  const int32_t* n_tile_active;       // [n_loops * n_requests]
  int32_t* skip;                      // [n_requests]: 1 = request refused (error bit 1)
  int32_t* err;
};
cudaError_t launch_append_batch_prep(const AppendBatchArgs& a, cudaStream_t stream);

// Launches one codec stage (kMode*) for a batch or a single request; a batch
// first plans its items into prefix_ws ([n_requests + 1] int32, device).
cudaError_t launch_codec(const CodecArgs& a, int mode, int32_t* prefix_ws, int sms, cudaStream_t stream);

// Quantise one value against its group's FP32 min and scale (scale 0: constant group).
__device__ __forceinline__ int quantize(float x, float mn, float s32) {
  if (s32 == 0.0f) return 0;
  float r = rintf(__fdiv_rn(__fsub_rn(x, mn), s32));
  r = fminf(fmaxf(r, 0.0f), 15.0f);
  return int(r);
}

}  // namespace kvq
