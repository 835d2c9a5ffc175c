/*
 * kvq_oracle.c — scalar CPU oracle for the FlashLoop packed-KV path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link,
 * load or execute this file or the library built from it: only tests/,
 * __graft_entry__.smoke() and the cpu_baseline / reference leg of bench.py use
 * it. It shares no source with the CUDA path (own format indexing, own
 * FP16/BF16 rounding written from IEEE-754, own group loops).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 *        (no SIMD intrinsics, no FMA contraction, IEEE single precision).
 *
 * Sources ("RFC" = "[RFC]: FlashLoop integration — token-sparse prefill,
 * sparse decode attention, and KV residual quantization", vllm-rlt issue #156;
 * "PR" = "INT4 KV packing/unpacking and cross-loop residual reconstruction",
 * vllm-rlt pull #166):
 *   - residual chain X̂1 = deq(q(X1)), δr = Xr − X̂(r−1), X̂r = X̂(r−1) + deq(q(δr)),
 *     subtracting the reconstructed predecessor:            RFC §3.3 (first two paragraphs)
 *   - affine INT4 group: scale = (max−min)/15, code = rounded/clipped
 *     (x−min)/scale, decode = min + scale·code; constant groups explicit;
 *     group size 64; FP16 params; K across token rows per channel, V across
 *     channels per token; BF16 compute dtype:               RFC §3.3 (third paragraph)
 *   - codes computed in FP32 before the FP16 metadata is rounded; nibble
 *     order; compact-row K groups for sparse residuals:      PR, review by 0z5a
 *   - two codes per uint8, FP16 min and scale, partial groups supported,
 *     subtraction/addition in the input compute dtype:       PR, "Purpose"
 *   - compact sparse residual rows, explicit logical→compact maps, absent
 *     residual = inherit (not code 0); loop-4 read example:  RFC §3.3 (fourth paragraph)
 *   - decode attention at the requested depth, scale 1/sqrt(head_dim):
 *                                                           RFC §3.2
 *   - K groups that never mix rows of different logical groups, so a page's
 *     metadata stays local (the alternative to compact-row groups):
 *                                                           PR, review by 0z5a (group ownership)
 *
 * Readings taken where the pages are silent (each also listed in the design doc):
 *   - code rounding: round half to even, then clamp to [0, 15];
 *   - division: IEEE-correct FP32 '/', no reciprocal;
 *   - constant group (max == min): scale stored as +0, every code 0, min
 *     stored as RN16(min); decoding gives min16;
 *   - nibble order: the even channel sits in the low nibble;
 *   - packing axis: channel pairs within one (row, head);
 *   - dequantisation rounds to BF16: RN_bf16(RN32(min16 + RN32(scale16·c)));
 *     each chain addition rounds to BF16: RN_bf16(RN32(X̂ + deq));
 *   - residual: δ = RN_bf16(RN32(X_r − X̂_{r−1})) at the stored rows;
 *   - GQA head mapping kv_head = q_head / (Hq / H);
 *   - the attention reference decodes the packed chain in FP32 (decode and
 *     chain sums rounded to FP32 only) before FP32 attention: the direct
 *     packed reader's values; the BF16 reconstruction is a separate output;
 *   - plane layout (head-major): codes u8[H][n][D/2]; K params f16[H][⌈n/G⌉][D];
 *     V params f16[H][n][⌈D/G⌉]; sparse index int32[n] ascending;
 *   - NVFP4 residual (orc_encode_nvfp4): two-level scaling in the order given
 *     there (tensor amax/2688, E4M3 block scale of amax_b/(6·s_t), E2M1 codes
 *     of δ/(s_b·s_t)); blocks of 16 channels of one (row, head) for K and V;
 *     the base stays INT4;
 *   - tile-local K grouping (ORC_KGROUP_TILE): a K group of a sparse loop holds
 *     the stored rows whose logical positions lie in one logical tile
 *     [G·k, G·k + G); its params sit in slot k of f16[H][⌈T/G⌉][D]; a tile with
 *     no stored row keeps +0 min and +0 scale (an empty stream stores no params).
 *     Dense loops group the same rows either way, so their bytes do not depend
 *     on the grouping.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_KIND_K 0
#define ORC_KIND_V 1

#define ORC_KGROUP_COMPACT 0 /* K groups: G consecutive stored rows */
#define ORC_KGROUP_TILE 1    /* K groups: the stored rows of one logical tile of G tokens */

#define ORC_FMT_INT4 0  /* affine INT4 groups of G (FP16 min and scale) */
#define ORC_FMT_NVFP4 1 /* E2M1 + E4M3 per 16 channels + FP32 per stream */

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENOMEM (-2)

/* ------------------------------------------------------------------------ */
/* IEEE-754 conversions, written from the binary16 / bfloat16 definitions.   */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return u;
}

static float bits_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* binary32 -> binary16, round to nearest, ties to even. Overflow gives ±inf,
 * underflow goes through the binary16 subnormal range, NaN stays NaN. */
uint16_t orc_f32_to_f16(float f) {
  uint32_t x = f32_bits(f);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t exp = (x >> 23) & 0xFFu;
  uint32_t man = x & 0x7FFFFFu;
  if (exp == 0xFFu) {
    if (man != 0) return (uint16_t)(sign | 0x7E00u);
    return (uint16_t)(sign | 0x7C00u);
  }
  if (exp == 0) return (uint16_t)sign; /* |f| < 2^-126: far below half of the smallest f16 subnormal */
  int e16 = (int)exp - 127 + 15;
  if (e16 >= 31) return (uint16_t)(sign | 0x7C00u);
  if (e16 <= 0) {
    /* Result is a binary16 subnormal m * 2^-24 (or rounds up to the smallest normal).
     * The binary32 significand with its hidden bit is sig * 2^(exp-150);
     * m = sig * 2^(exp-150+24) = sig >> (126 - exp). */
    int shift = 126 - (int)exp;
    if (shift > 24) return (uint16_t)sign; /* |f| < 2^-25: rounds to zero */
    uint32_t sig = man | 0x800000u;
    uint32_t m = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (m & 1u))) m += 1u;
    return (uint16_t)(sign | m);
  }
  uint32_t h = sign | ((uint32_t)e16 << 10) | (man >> 13);
  uint32_t rem = man & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u; /* a carry may roll into the exponent (and to inf) */
  return (uint16_t)h;
}

float orc_f16_to_f32(uint16_t h) {
  uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
  uint32_t exp = ((uint32_t)h >> 10) & 0x1Fu;
  uint32_t man = (uint32_t)h & 0x3FFu;
  if (exp == 0x1Fu) return bits_f32(sign | 0x7F800000u | (man << 13));
  if (exp == 0) {
    /* zero or subnormal: man * 2^-24, exact in binary32 */
    float v = (float)man * 5.9604644775390625e-8f; /* 2^-24 */
    return sign ? -v : v;
  }
  return bits_f32(sign | ((exp - 15u + 127u) << 23) | (man << 13));
}

/* binary32 -> bfloat16 (the upper half of binary32), round to nearest, ties to even. */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t x = f32_bits(f);
  if ((x & 0x7F800000u) == 0x7F800000u && (x & 0x7FFFFFu) != 0) return (uint16_t)((x >> 16) | 0x0040u);
  uint32_t hi = x >> 16;
  uint32_t rem = x & 0xFFFFu;
  if (rem > 0x8000u || (rem == 0x8000u && (hi & 1u))) hi += 1u;
  return (uint16_t)hi;
}

float orc_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/* Batch forms of the conversions, for the tests that pin them. */
void orc_f32_to_f16_n(const float* x, uint16_t* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_f16(x[i]);
}
void orc_f32_to_bf16_n(const float* x, uint16_t* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_bf16(x[i]);
}
void orc_f16_to_f32_n(const uint16_t* x, float* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_f16_to_f32(x[i]);
}

/* Round half to even for 0 <= v < 2^22 (the quantiser's ratio lies in [0, 15]). */
static float round_half_even(float v) {
  float fl = floorf(v);
  float frac = v - fl; /* exact: both lie in the same binade range below 2^23 */
  if (frac > 0.5f) return fl + 1.0f;
  if (frac < 0.5f) return fl;
  return (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 and FP4 E2M1 (the NVFP4 element and block-scale types; codec PR  */
/* review by 0z5a: "E2M1 round-to-nearest-even, E4M3 scale rounding").       */
/* ------------------------------------------------------------------------ */

/* E4M3, finite variant: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
 * infinities; largest finite 448 = 1.75·2^8; subnormals m·2^-9. Round to
 * nearest, ties to even; anything above 448 saturates to 448. */
uint8_t orc_f32_to_e4m3(float f) {
  uint8_t sign = (f32_bits(f) >> 31) ? 0x80 : 0x00;
  float v = fabsf(f);
  if (v != v) return 0x7F; /* NaN */
  if (v >= 448.0f) return (uint8_t)(sign | (15 << 3) | 6);
  if (v < 0.015625f) { /* below 2^-6: subnormal, in units of 2^-9 */
    float m = round_half_even(v * 512.0f);
    if (m >= 8.0f) return (uint8_t)(sign | (1 << 3)); /* rounds up to 2^-6 */
    return (uint8_t)(sign | (int)m);
  }
  int ex;
  float fr = frexpf(v, &ex); /* v = fr·2^ex, fr in [0.5, 1) */
  int E = ex - 1;            /* v = (2 fr)·2^E, 2 fr in [1, 2) */
  float M = round_half_even((2.0f * fr - 1.0f) * 8.0f);
  if (M >= 8.0f) {
    M = 0.0f;
    E += 1;
  }
  if (E > 8 || (E == 8 && M > 6.0f)) return (uint8_t)(sign | (15 << 3) | 6);
  return (uint8_t)(sign | ((E + 7) << 3) | (int)M);
}

float orc_e4m3_to_f32(uint8_t b) {
  int E = (b >> 3) & 15, M = b & 7;
  float v = (E == 0) ? ldexpf((float)M, -9) : ldexpf(1.0f + (float)M / 8.0f, E - 7);
  return (b & 0x80) ? -v : v;
}

/* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; the eight magnitudes
 * below, code = index. The nearest magnitude wins; a tie goes to the even
 * code (even mantissa); anything above 6 saturates to 6. The sign is kept,
 * zero included. */
static const float kE2M1[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

uint8_t orc_f32_to_e2m1(float f) {
  uint8_t sign = (f32_bits(f) >> 31) ? 0x8 : 0x0;
  float v = fabsf(f);
  int best = 7;
  if (v <= 6.0f) {
    best = 0;
    for (int k = 1; k < 8; ++k) {
      float dk = fabsf(v - kE2M1[k]), db = fabsf(v - kE2M1[best]);
      if (dk < db || (dk == db && (k % 2) == 0)) best = k;
    }
  }
  return (uint8_t)(sign | best);
}

float orc_e2m1_to_f32(uint8_t n) {
  float v = kE2M1[n & 7];
  return (n & 8) ? -v : v;
}

void orc_f32_to_e4m3_n(const float* x, uint8_t* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_e4m3(x[i]);
}
void orc_f32_to_e2m1_n(const float* x, uint8_t* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_e2m1(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Affine INT4 group quantiser (RFC §3.3; FP32 codes before FP16 rounding,    */
/* PR review by 0z5a).                                                        */
/* ------------------------------------------------------------------------ */

/* Quantise n values v[0], v[step], ... (each a BF16 value widened to FP32).
 * Writes n codes in [0, 15] to code[0..n-1] and the FP16 min and scale. */
static void quantize_group(const float* v, int n, int step, uint8_t* code, uint16_t* min16, uint16_t* scale16) {
  float mn = v[0], mx = v[0];
  for (int i = 1; i < n; ++i) {
    float x = v[(int64_t)i * step];
    if (x < mn) mn = x;
    if (x > mx) mx = x;
  }
  *min16 = orc_f32_to_f16(mn);
  if (mx == mn) { /* constant group: defined explicitly, no division */
    *scale16 = orc_f32_to_f16(0.0f);
    for (int i = 0; i < n; ++i) code[i] = 0;
    return;
  }
  float range = mx - mn;      /* RN32 */
  float s32 = range / 15.0f;  /* RN32, IEEE division */
  *scale16 = orc_f32_to_f16(s32);
  for (int i = 0; i < n; ++i) {
    float x = v[(int64_t)i * step];
    float diff = x - mn;      /* RN32, >= 0 */
    float ratio = diff / s32; /* RN32, IEEE division */
    float r = round_half_even(ratio);
    if (r < 0.0f) r = 0.0f;
    if (r > 15.0f) r = 15.0f;
    code[i] = (uint8_t)r;
  }
}

/* Decode one code: RN_bf16(RN32(f32(min16) + RN32(f32(scale16) * c))). */
static float dequant(uint16_t min16, uint16_t scale16, int c) {
  float m = orc_f16_to_f32(min16);
  float s = orc_f16_to_f32(scale16);
  float prod = s * (float)c;
  float sum = m + prod;
  return orc_bf16_to_f32(orc_f32_to_bf16(sum));
}

/* ------------------------------------------------------------------------ */
/* Plane geometry (head-major).                                              */
/* ------------------------------------------------------------------------ */

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* K groups per head of a stream: by stored rows, or one per logical tile of a
 * tile-grouped sparse stream. */
static int64_t k_groups(int n, int T, int G, int kgroup, int sparse) {
  if (n <= 0) return 0; /* an empty stream stores no params */
  return (kgroup == ORC_KGROUP_TILE && sparse) ? ceil_div(T, G) : ceil_div(n, G);
}

/* Byte-exact sizes of the planes of one stream with n stored rows of T tokens. */
int64_t orc_codes_bytes(int n, int H, int D) { return (int64_t)H * n * (D / 2); }
int64_t orc_param_count_ex(int kind, int n, int T, int H, int D, int G, int kgroup, int sparse) {
  if (kind == ORC_KIND_K) return (int64_t)H * k_groups(n, T, G, kgroup, sparse) * D;
  return (int64_t)H * n * ceil_div(D, G);
}
int64_t orc_param_count(int kind, int n, int H, int D, int G) {
  return orc_param_count_ex(kind, n, n, H, D, G, ORC_KGROUP_COMPACT, 0);
}
int64_t orc_stream_bytes_ex(int kind, int n, int T, int H, int D, int G, int kgroup, int sparse) {
  return orc_codes_bytes(n, H, D) + 2 * 2 * orc_param_count_ex(kind, n, T, H, D, G, kgroup, sparse) +
         (sparse ? 4 * (int64_t)n : 0);
}
int64_t orc_stream_bytes(int kind, int n, int H, int D, int G, int sparse) {
  return orc_stream_bytes_ex(kind, n, n, H, D, G, ORC_KGROUP_COMPACT, sparse);
}
/* NVFP4 stream: E2M1 codes, one E4M3 byte per 16 channels, the FP32 tensor scale. */
int64_t orc_stream_bytes_nvfp4(int n, int H, int D, int sparse) {
  if (n <= 0) return 0;
  return orc_codes_bytes(n, H, D) + (int64_t)H * n * (D / 16) + 4 + (sparse ? 4 * (int64_t)n : 0);
}

static int64_t code_byte_index(int n, int D, int h, int row, int d) {
  return ((int64_t)h * n + row) * (D / 2) + d / 2;
}
/* Params of (head h, stored row, channel d). K: group kg of ngk groups per head
 * (the caller maps the row to its group); V: the row's channel group. */
static int64_t k_param_index(int64_t ngk, int D, int h, int64_t kg, int d) { return ((int64_t)h * ngk + kg) * D + d; }
static int64_t v_param_index(int n, int D, int G, int h, int row, int d) {
  return ((int64_t)h * n + row) * ceil_div(D, G) + d / G;
}

static int get_code(const uint8_t* codes, int n, int D, int h, int row, int d) {
  uint8_t b = codes[code_byte_index(n, D, h, row, d)];
  return (d & 1) ? (b >> 4) : (b & 0x0F);
}

/* An ascending, duplicate-free index list inside [0, T). */
static int check_active(const int32_t* a, int n, int T) {
  for (int i = 0; i < n; ++i) {
    if (a[i] < 0 || a[i] >= T) return 0;
    if (i > 0 && a[i] <= a[i - 1]) return 0;
  }
  return 1;
}

/* ------------------------------------------------------------------------ */
/* Encode one stream.                                                        */
/* ------------------------------------------------------------------------ */

/*
 * x    : BF16 bits [T][H][D], the loop-r source in logical token order.
 * pred : BF16 bits [T][H][D], X̂_{r-1} in logical order; NULL encodes the base (loop 1).
 * active, n : sorted logical rows to store (NULL: dense, n must equal T).
 * kgroup : ORC_KGROUP_COMPACT or ORC_KGROUP_TILE (K only; V ignores it).
 * Outputs use the head-major planes described at the top of the file.
 */
int orc_encode_ex(int kind, int T, int H, int D, int G, int kgroup, const uint16_t* x, const uint16_t* pred,
                  const int32_t* active, int n, uint8_t* codes, uint16_t* mins, uint16_t* scales) {
  if (T < 0 || H <= 0 || D <= 0 || (D & 1) || G <= 0) return ORC_EINVAL;
  if (kind != ORC_KIND_K && kind != ORC_KIND_V) return ORC_EINVAL;
  if (kgroup != ORC_KGROUP_COMPACT && kgroup != ORC_KGROUP_TILE) return ORC_EINVAL;
  if (active == NULL) {
    if (n != T) return ORC_EINVAL;
  } else if (n < 0 || n > T || !check_active(active, n, T)) {
    return ORC_EINVAL;
  }
  if (n == 0) return ORC_OK;

  /* Values to quantise, in compact row order: v[row][h][d] (FP32 from BF16). */
  float* v = (float*)malloc(sizeof(float) * (size_t)n * H * D);
  uint8_t* c = (uint8_t*)malloc((size_t)n * H * D);
  if (!v || !c) {
    free(v);
    free(c);
    return ORC_ENOMEM;
  }
  for (int row = 0; row < n; ++row) {
    int t = active ? active[row] : row;
    for (int h = 0; h < H; ++h) {
      for (int d = 0; d < D; ++d) {
        int64_t li = ((int64_t)t * H + h) * D + d;
        float xv = orc_bf16_to_f32(x[li]);
        float val;
        if (pred == NULL) {
          val = xv;
        } else {
          float diff = xv - orc_bf16_to_f32(pred[li]); /* RN32 */
          val = orc_bf16_to_f32(orc_f32_to_bf16(diff)); /* residual in the BF16 compute dtype */
        }
        v[((int64_t)row * H + h) * D + d] = val;
      }
    }
  }

  if (kind == ORC_KIND_K) {
    /* K: per (head, channel), groups of stored rows. Compact grouping: G
     * consecutive stored rows. Tile grouping of a sparse loop: the stored rows
     * of logical tile k (consecutive too, the index being ascending), group k. */
    int tiled = (kgroup == ORC_KGROUP_TILE && active != NULL);
    int64_t ng = k_groups(n, T, G, kgroup, active != NULL);
    int32_t* first = (int32_t*)malloc(sizeof(int32_t) * (size_t)(ng + 1));
    if (!first) {
      free(v);
      free(c);
      return ORC_ENOMEM;
    }
    for (int64_t g = 0; g <= ng; ++g) {
      if (!tiled) {
        first[g] = (int32_t)(g * G < n ? g * G : n);
      } else { /* first stored row at or after logical token G·g */
        int r = 0;
        while (r < n && active[r] < g * G) ++r;
        first[g] = r;
      }
    }
    uint8_t gc[4096];
    for (int h = 0; h < H; ++h) {
      for (int d = 0; d < D; ++d) {
        for (int64_t g = 0; g < ng; ++g) {
          int r0 = first[g];
          int len = first[g + 1] - r0;
          int64_t pi = k_param_index(ng, D, h, g, d);
          if (len == 0) { /* a tile with no stored row */
            mins[pi] = 0;
            scales[pi] = 0;
            continue;
          }
          const float* base = v + ((int64_t)r0 * H + h) * D + d;
          uint16_t m16, s16;
          quantize_group(base, len, H * D, gc, &m16, &s16);
          for (int i = 0; i < len; ++i) c[((int64_t)(r0 + i) * H + h) * D + d] = gc[i];
          mins[pi] = m16;
          scales[pi] = s16;
        }
      }
    }
    free(first);
  } else {
    /* V: per (stored row, head), groups of G consecutive channels. */
    int ngc = (int)ceil_div(D, G);
    uint8_t gc[4096];
    for (int row = 0; row < n; ++row) {
      for (int h = 0; h < H; ++h) {
        for (int k = 0; k < ngc; ++k) {
          int d0 = k * G;
          int len = (d0 + G <= D) ? G : D - d0;
          const float* base = v + ((int64_t)row * H + h) * D + d0;
          uint16_t m16, s16;
          quantize_group(base, len, 1, gc, &m16, &s16);
          for (int i = 0; i < len; ++i) c[((int64_t)row * H + h) * D + d0 + i] = gc[i];
          int64_t pi = v_param_index(n, D, G, h, row, d0);
          mins[pi] = m16;
          scales[pi] = s16;
        }
      }
    }
  }

  /* Pack: byte (h, row, k) = code(row, h, 2k) | code(row, h, 2k+1) << 4. */
  for (int h = 0; h < H; ++h) {
    for (int row = 0; row < n; ++row) {
      for (int k = 0; k < D / 2; ++k) {
        uint8_t lo = c[((int64_t)row * H + h) * D + 2 * k];
        uint8_t hi = c[((int64_t)row * H + h) * D + 2 * k + 1];
        codes[code_byte_index(n, D, h, row, 2 * k)] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
  free(v);
  free(c);
  return ORC_OK;
}

int orc_encode(int kind, int T, int H, int D, int G, const uint16_t* x, const uint16_t* pred, const int32_t* active,
               int n, uint8_t* codes, uint16_t* mins, uint16_t* scales) {
  return orc_encode_ex(kind, T, H, D, G, ORC_KGROUP_COMPACT, x, pred, active, n, codes, mins, scales);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 residual (codec PR review by 0z5a: E2M1 elements, one E4M3 scale per */
/* 16 elements, one FP32 scale per tensor; symmetric, no zero point; blocks   */
/* along channels for K and V alike, so K metadata is page-local).           */
/* ------------------------------------------------------------------------ */

/*
 * Encode the residual of loop r as NVFP4 (a residual only: the base stays INT4).
 * Same residual rows as orc_encode: δ = RN_bf16(RN32(X_r − X̂_{r−1})) at the
 * stored rows. Two-level scaling, in this order:
 *   a_t  = max |δ| over the whole stream (all stored rows, heads, channels);
 *   s_t  = RN32(a_t / 2688)                     FP32 tensor scale (2688 = 6·448)
 *   per block of 16 channels of one (row, head), a_b = max |δ| in the block:
 *   s_b  = E4M3(RN32(a_b / RN32(6·s_t)))        block scale (a_t's block: 448)
 *   e_b  = RN32(f32(s_b)·s_t)                   the block's quantisation step
 *   code = E2M1(RN32(δ / e_b)) (IEEE division; e_b = 0: code +0)
 * a_t = 0 gives s_t = 0 and every scale and code 0.
 * Decode: RN32(RN32(e2m1·s_b)·s_t) (e2m1·s_b is exact); the BF16 chain rounds it
 * to BF16 before the add, as for INT4.
 * Planes: codes u8[H][n][D/2] (nibble = code, even channel low);
 * bscale u8[H][n][D/16] (E4M3 bits); *tscale = s_t.
 */
int orc_encode_nvfp4(int kind, int T, int H, int D, const uint16_t* x, const uint16_t* pred, const int32_t* active,
                     int n, uint8_t* codes, uint8_t* bscale, float* tscale) {
  if (T < 0 || H <= 0 || D <= 0 || (D % 16) != 0 || pred == NULL) return ORC_EINVAL;
  if (kind != ORC_KIND_K && kind != ORC_KIND_V) return ORC_EINVAL;
  if (active == NULL) {
    if (n != T) return ORC_EINVAL;
  } else if (n < 0 || n > T || !check_active(active, n, T)) {
    return ORC_EINVAL;
  }
  *tscale = 0.0f;
  if (n == 0) return ORC_OK;
  float* v = (float*)malloc(sizeof(float) * (size_t)n * H * D);
  if (!v) return ORC_ENOMEM;
  float amax = 0.0f;
  for (int row = 0; row < n; ++row) {
    int t = active ? active[row] : row;
    for (int h = 0; h < H; ++h)
      for (int d = 0; d < D; ++d) {
        int64_t li = ((int64_t)t * H + h) * D + d;
        float diff = orc_bf16_to_f32(x[li]) - orc_bf16_to_f32(pred[li]); /* RN32 */
        float val = orc_bf16_to_f32(orc_f32_to_bf16(diff));
        v[((int64_t)row * H + h) * D + d] = val;
        if (fabsf(val) > amax) amax = fabsf(val);
      }
  }
  float st = amax / 2688.0f; /* RN32 */
  *tscale = st;
  float six_st = 6.0f * st;  /* RN32 */
  for (int row = 0; row < n; ++row)
    for (int h = 0; h < H; ++h) {
      const float* r = v + ((int64_t)row * H + h) * D;
      uint8_t* crow = codes + ((int64_t)h * n + row) * (D / 2);
      for (int b = 0; b < D / 16; ++b) {
        float ab = 0.0f;
        for (int i = 0; i < 16; ++i)
          if (fabsf(r[16 * b + i]) > ab) ab = fabsf(r[16 * b + i]);
        uint8_t sb = (amax == 0.0f) ? 0 : orc_f32_to_e4m3(ab / six_st);
        bscale[((int64_t)h * n + row) * (D / 16) + b] = sb;
        float eb = orc_e4m3_to_f32(sb) * st; /* RN32 */
        for (int i = 0; i < 16; i += 2) {
          uint8_t c[2];
          for (int k = 0; k < 2; ++k)
            c[k] = (eb == 0.0f) ? 0 : orc_f32_to_e2m1(r[16 * b + i + k] / eb); /* IEEE division, RN32 */
          crow[(16 * b + i) / 2] = (uint8_t)(c[0] | (c[1] << 4));
        }
      }
    }
  free(v);
  return ORC_OK;
}

/* Decode one NVFP4 element in FP32: RN32(RN32(e2m1 · s_b) · s_t). */
static float nvfp4_dequant(uint8_t code, uint8_t sb, float st) {
  float p = orc_e2m1_to_f32(code) * orc_e4m3_to_f32(sb); /* exact */
  return p * st;
}

/* ------------------------------------------------------------------------ */
/* Reconstruct the chain to a requested depth (RFC §3.3).                     */
/* ------------------------------------------------------------------------ */

typedef struct {
  int32_t n;              /* stored rows */
  int32_t kgroup;         /* ORC_KGROUP_COMPACT or ORC_KGROUP_TILE */
  const int32_t* active;  /* NULL: dense (n == T) */
  const uint8_t* codes;
  const uint16_t* mins;   /* INT4 */
  const uint16_t* scales; /* INT4 */
  int32_t fmt;            /* ORC_FMT_INT4 or ORC_FMT_NVFP4 (residual loops only) */
  int32_t _pad;
  const uint8_t* bscale;  /* NVFP4: E4M3 [H][n][D/16] */
  const float* tscale;    /* NVFP4: the FP32 tensor scale */
} orc_stream;

/* Index of the params of (head h, stored row, channel d) of stream s. */
static int64_t stream_param_index(int kind, const orc_stream* s, int T, int D, int G, int h, int row, int d) {
  if (kind != ORC_KIND_K) return v_param_index(s->n, D, G, h, row, d);
  int sparse = s->active != NULL;
  int64_t ng = k_groups(s->n, T, G, s->kgroup, sparse);
  int64_t kg = (s->kgroup == ORC_KGROUP_TILE && sparse) ? s->active[row] / G : row / G;
  return k_param_index(ng, D, h, kg, d);
}

/* Decoded value (FP32, before any BF16 rounding) of (head h, stored row, channel d)
 * of stream s: INT4 RN32(min16 + RN32(scale16·c)), or the NVFP4 decode. */
static float stream_dequant32(int kind, const orc_stream* s, int T, int D, int G, int h, int row, int d) {
  int c = get_code(s->codes, s->n, D, h, row, d);
  if (s->fmt == ORC_FMT_NVFP4)
    return nvfp4_dequant((uint8_t)c, s->bscale[((int64_t)h * s->n + row) * (D / 16) + d / 16], s->tscale[0]);
  int64_t pi = stream_param_index(kind, s, T, D, G, h, row, d);
  float m = orc_f16_to_f32(s->mins[pi]);
  float sc = orc_f16_to_f32(s->scales[pi]);
  float prod = sc * (float)c;
  return m + prod;
}


/*
 * loops[0] is the base, loops[j-1] the residual of loop j. out: BF16 bits
 * [T][H][D] in logical order. A token absent from loop j keeps its value
 * (inheritance); it is never decoded from a code.
 */
int orc_reconstruct(int kind, int T, int H, int D, int G, int depth, const orc_stream* loops, uint16_t* out) {
  if (T < 0 || H <= 0 || D <= 0 || (D & 1) || G <= 0 || depth < 1) return ORC_EINVAL;
  if (loops[0].active != NULL || loops[0].n != T || loops[0].fmt != ORC_FMT_INT4) return ORC_EINVAL;
  for (int j = 1; j < depth; ++j) {
    if (loops[j].active == NULL) {
      if (loops[j].n != T) return ORC_EINVAL;
    } else if (loops[j].n < 0 || loops[j].n > T || !check_active(loops[j].active, loops[j].n, T)) {
      return ORC_EINVAL;
    }
  }
  int32_t* rowmap = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
  if (!rowmap) return ORC_ENOMEM;

  /* Base. */
  const orc_stream* b = &loops[0];
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      for (int d = 0; d < D; ++d) {
        int64_t pi = stream_param_index(kind, b, T, D, G, h, t, d);
        float val = dequant(b->mins[pi], b->scales[pi], get_code(b->codes, T, D, h, t, d));
        out[((int64_t)t * H + h) * D + d] = orc_f32_to_bf16(val);
      }

  /* Residual loops 2..depth. */
  for (int j = 1; j < depth; ++j) {
    const orc_stream* s = &loops[j];
    for (int t = 0; t < T; ++t) rowmap[t] = -1;
    for (int i = 0; i < s->n; ++i) rowmap[s->active ? s->active[i] : i] = i;
    for (int t = 0; t < T; ++t) {
      int row = rowmap[t];
      if (row < 0) continue; /* absent: inherit */
      for (int h = 0; h < H; ++h)
        for (int d = 0; d < D; ++d) {
          /* the decoded residual in the BF16 compute dtype (INT4: RN_bf16(min16 + scale16·c)) */
          float dq = orc_bf16_to_f32(orc_f32_to_bf16(stream_dequant32(kind, s, T, D, G, h, row, d)));
          int64_t li = ((int64_t)t * H + h) * D + d;
          float sum = orc_bf16_to_f32(out[li]) + dq; /* RN32 */
          out[li] = orc_f32_to_bf16(sum);
        }
    }
  }
  free(rowmap);
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* FP32 decode of the packed chain: the values a direct packed reader sees.  */
/* ------------------------------------------------------------------------ */

/*
 * Same chain as orc_reconstruct, evaluated in FP32 without BF16 rounding:
 * decode = RN32(f32(min16) + RN32(f32(scale16) * c)) and each present loop is
 * added with one FP32 rounding; absent tokens inherit. This is the reference
 * of the attention reader, which consumes the packed planes directly (RFC §3.3)
 * and is compared in FP32 on the same packed data; its distance to the BF16
 * reconstruction is the direct-reader error that RFC §9 asks to bound.
 * out: FP32 [T][H][D].
 */
int orc_decode_f32(int kind, int T, int H, int D, int G, int depth, const orc_stream* loops, float* out) {
  if (T < 0 || H <= 0 || D <= 0 || (D & 1) || G <= 0 || depth < 1) return ORC_EINVAL;
  if (loops[0].active != NULL || loops[0].n != T || loops[0].fmt != ORC_FMT_INT4) return ORC_EINVAL;
  for (int j = 1; j < depth; ++j) {
    if (loops[j].active == NULL) {
      if (loops[j].n != T) return ORC_EINVAL;
    } else if (loops[j].n < 0 || loops[j].n > T || !check_active(loops[j].active, loops[j].n, T)) {
      return ORC_EINVAL;
    }
  }
  int32_t* rowmap = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
  if (!rowmap) return ORC_ENOMEM;
  for (int j = 0; j < depth; ++j) {
    const orc_stream* s = &loops[j];
    for (int t = 0; t < T; ++t) rowmap[t] = -1;
    for (int i = 0; i < s->n; ++i) rowmap[s->active ? s->active[i] : i] = i;
    for (int t = 0; t < T; ++t) {
      int row = rowmap[t];
      if (row < 0) continue;
      for (int h = 0; h < H; ++h)
        for (int d = 0; d < D; ++d) {
          float dq = stream_dequant32(kind, s, T, D, G, h, row, d);
          int64_t li = ((int64_t)t * H + h) * D + d;
          out[li] = (j == 0) ? dq : out[li] + dq;
        }
    }
  }
  free(rowmap);
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Decode attention in FP32 (RFC §3.2, §5).                                   */
/* ------------------------------------------------------------------------ */

/*
 * q: BF16 bits [Hq][D]; khat, vhat: BF16 bits [T][H][D]; out: FP32 [Hq][D].
 * One query token attends to all T stored tokens (no mask: in decode the
 * query follows every stored position). kv_head = q_head / (Hq / H).
 * s_t = (sum_d q_d k_td, in channel order) * scale; p_t = exp(s_t - max s);
 * o_d = (sum_t p_t v_td, in token order) / (sum_t p_t).
 */
static int attention_core(int T, int H, int Hq, int D, const uint16_t* q, const float* kf, const float* vf,
                          float scale, float* out) {
  if (T <= 0 || H <= 0 || Hq <= 0 || D <= 0 || Hq % H != 0) return ORC_EINVAL;
  int g = Hq / H;
  float* s = (float*)malloc(sizeof(float) * (size_t)T);
  float* acc = (float*)malloc(sizeof(float) * (size_t)D);
  if (!s || !acc) {
    free(s);
    free(acc);
    return ORC_ENOMEM;
  }
  for (int hq = 0; hq < Hq; ++hq) {
    int h = hq / g;
    float mx = -INFINITY;
    for (int t = 0; t < T; ++t) {
      float dot = 0.0f;
      for (int d = 0; d < D; ++d) {
        float prod = orc_bf16_to_f32(q[(int64_t)hq * D + d]) * kf[((int64_t)t * H + h) * D + d];
        dot = dot + prod;
      }
      s[t] = dot * scale;
      if (s[t] > mx) mx = s[t];
    }
    float L = 0.0f;
    for (int d = 0; d < D; ++d) acc[d] = 0.0f;
    for (int t = 0; t < T; ++t) {
      float p = expf(s[t] - mx);
      L = L + p;
      for (int d = 0; d < D; ++d) {
        float prod = p * vf[((int64_t)t * H + h) * D + d];
        acc[d] = acc[d] + prod;
      }
    }
    for (int d = 0; d < D; ++d) out[(int64_t)hq * D + d] = acc[d] / L;
  }
  free(s);
  free(acc);
  return ORC_OK;
}

/*
 * q: BF16 bits [Hq][D]; khat, vhat: BF16 bits [T][H][D]; out: FP32 [Hq][D].
 * One query token attends to all T stored tokens (no mask: in decode the
 * query follows every stored position). kv_head = q_head / (Hq / H).
 * s_t = (sum_d q_d k_td, in channel order) * scale; p_t = exp(s_t - max s);
 * o_d = (sum_t p_t v_td, in token order) / (sum_t p_t).
 */
int orc_attention(int T, int H, int Hq, int D, const uint16_t* q, const uint16_t* khat, const uint16_t* vhat,
                  float scale, float* out) {
  if (T <= 0 || H <= 0 || D <= 0) return ORC_EINVAL;
  size_t n = (size_t)T * H * D;
  float* kf = (float*)malloc(sizeof(float) * n);
  float* vf = (float*)malloc(sizeof(float) * n);
  if (!kf || !vf) {
    free(kf);
    free(vf);
    return ORC_ENOMEM;
  }
  for (size_t i = 0; i < n; ++i) {
    kf[i] = orc_bf16_to_f32(khat[i]);
    vf[i] = orc_bf16_to_f32(vhat[i]);
  }
  int rc = attention_core(T, H, Hq, D, q, kf, vf, scale, out);
  free(kf);
  free(vf);
  return rc;
}

/* Same attention on FP32 K and V (the FP32 decode of the packed chain). */
int orc_attention_f32(int T, int H, int Hq, int D, const uint16_t* q, const float* kf, const float* vf, float scale,
                      float* out) {
  return attention_core(T, H, Hq, D, q, kf, vf, scale, out);
}
