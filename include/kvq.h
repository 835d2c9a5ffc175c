/*
 * kvq.h — C ABI of libkvq.so: the FlashLoop packed-KV hot path on one GB300
 * (sm_103a). INT4 base + cross-loop residual codec, residual-chain
 * reconstruction, and packed-KV GQA decode attention.
 *
 * Pages cited ("RFC" = "[RFC]: FlashLoop integration — token-sparse prefill,
 * sparse decode attention, and KV residual quantization", vllm-rlt issue #156;
 * "codec PR" = "INT4 KV packing/unpacking and cross-loop residual
 * reconstruction", vllm-rlt pull #166).
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers owned by the caller. The library
 *     allocates no device memory and keeps no pointer after a call returns.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous: a call returns before the GPU finishes. No
 *     call reads device data back to the host or synchronises (RFC §6.2).
 *   - Arguments are checked on the host before anything is launched. A bad
 *     argument returns a negative kvq_status and launches nothing; there is no
 *     CPU fallback and no other backend (RFC §4: fail clearly).
 *     kvq_last_error() gives a one-line reason for the last failure on the
 *     calling thread.
 *   - BF16 and FP16 values travel as their 16-bit patterns (uint16_t).
 *   - The GPU kernels support head_dim == 128 (other sizes: UNSUPPORTED).
 *
 * Packed format, version 1 (one stream = one loop of K or V of one
 * request/layer; RFC §3.3, codec PR "Purpose"):
 *   codes   uint8  [H][n_rows][D/2]   byte (h,i,k) = code(i,h,2k) | code(i,h,2k+1) << 4
 *   K mins, scales  FP16 [H][ceil(n_rows/64)][D]   one group = 64 consecutive stored
 *                                                  rows of one (head, channel)
 *                   (KVQ_KGROUP_TILE, sparse stream)
 *                   FP16 [H][ceil(n_tokens/64)][D] group k = the stored rows whose
 *                                                  logical token lies in [64k, 64k+64);
 *                                                  a tile with no stored row keeps
 *                                                  min +0 and scale +0
 *   V mins, scales  FP16 [H][n_rows][ceil(D/64)]   one group = 64 channels of one
 *                                                  (stored row, head)
 *   active_idx int32 [n_rows]  ascending logical rows of a compact sparse
 *                              residual; NULL for a dense stream (n_rows == n_tokens)
 *   tile_dir   int32 [ceil(n_tokens/64)+1]  tile_dir[k] = number of active
 *                              indices below 64k (derived map, see kvq_build_tile_dir)
 * Quantiser (RFC §3.3; codes from the FP32 scale, then FP16 metadata, codec
 * PR review by 0z5a): scale = RN32(RN32(max-min)/15); code =
 * clamp(rint_even(RN32(RN32(x-min)/scale)), 0, 15); a constant group stores
 * scale 0 and codes 0. Decode: RN_bf16(min16 + scale16*code). Residual loop r:
 * delta = RN_bf16(X_r - X̂_{r-1}) at the stored rows; X̂_r = RN_bf16(X̂_{r-1} +
 * decode(delta)) where a token is stored, and X̂_{r-1} (inherited) where it is
 * absent (RFC §3.3: an absent residual is not an INT4 code 0).
 *
 * NVFP4 residual format (codec PR review by 0z5a: "INT4 base plus NVFP4
 * residuals is a legitimate option"; E2M1 elements, one E4M3 scale per 16
 * elements, one FP32 scale per tensor). A residual stream (never the base) may
 * use format KVQ_FMT_NVFP4 (group 16) instead of KVQ_FMT_INT4 (group 64):
 *   codes   uint8 [H][n_rows][D/2]    byte = e2m1(2k) | e2m1(2k+1) << 4 (sign bit 3)
 *   mins    read as uint8 [H][n_rows][D/16]   E4M3 scale of each 16-channel block
 *                                             of one (stored row, head), K and V alike
 *   scales  read as float [4]         [0] the FP32 tensor scale s_t, [1] scratch of
 *                                     the encoder (the stream's max |delta|)
 * Encode of loop r, delta as above: s_t = RN32(max|delta| / 2688); block scale
 * s_b = E4M3(RN32(a_b / RN32(6 s_t))) (a_b = max |delta| of the block; E4M3
 * round to nearest even, saturating at 448); code = E2M1(RN32(delta /
 * RN32(s_b s_t))) (nearest of 0, .5, 1, 1.5, 2, 3, 4, 6, ties to even,
 * saturating at 6, sign kept; a zero step gives code 0). Decode:
 * RN32(RN32(e2m1 s_b) s_t), rounded to BF16 before the chain add like INT4.
 *
 * K grouping (codec PR review by 0z5a, group ownership vs pages): the codec
 * PR groups a sparse K residual over consecutive compact rows, so one group can
 * mix distant positions. KVQ_KGROUP_TILE keeps every K group inside one
 * 64-token logical tile instead, so a tile's rows and metadata can be freed,
 * moved or shared without re-encoding any other tile. Dense streams group the
 * same rows either way (identical bytes).
 *
 * Alignment: every plane pointer (codes, mins, scales, active_idx) must be
 * 16-byte aligned and its allocation at least kvq_plane_bytes() long (sizes
 * are rounded up to 16 bytes so the kernels can move whole 16-byte vectors).
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_FORMAT_VERSION 1u
#define KVQ_BITS 4
#define KVQ_GROUP 64
#define KVQ_TILE 64
#define KVQ_MAX_LOOPS 8
#define KVQ_NIBBLE_LO_FIRST 0
#define KVQ_KGROUP_COMPACT 0 /* K groups: 64 consecutive stored rows (default) */
#define KVQ_KGROUP_TILE 1    /* K groups: the stored rows of one 64-token logical tile */
#define KVQ_FMT_INT4 0       /* affine INT4 groups of 64 with FP16 min and scale */
#define KVQ_FMT_NVFP4 1      /* E2M1 + E4M3 per 16 channels + FP32 per stream (residual loops) */

typedef int32_t kvq_status;
#define KVQ_OK 0
#define KVQ_ERR_BAD_ARG (-1)     /* null pointer, size out of range, inconsistent descriptors */
#define KVQ_ERR_UNSUPPORTED (-2) /* valid format the kernels do not implement (e.g. head_dim != 128) */
#define KVQ_ERR_MISALIGNED (-3)  /* a plane pointer is not 16-byte aligned */
#define KVQ_ERR_WORKSPACE (-4)   /* workspace missing or smaller than required */
#define KVQ_ERR_CUDA (-5)        /* a CUDA runtime call or kernel launch failed */

/* Opaque CUDA stream handle: identical to cudaStream_t. */
typedef struct CUstream_st* kvq_cuda_stream;

enum { KVQ_K = 0, KVQ_V = 1 };
enum { KVQ_PLANE_CODES = 0, KVQ_PLANE_MINS = 1, KVQ_PLANE_SCALES = 2, KVQ_PLANE_INDEX = 3, KVQ_PLANE_TILE_DIR = 4 };

/* Descriptor of one stream (host memory; the pointers inside are device
 * pointers). The descriptor records format, grouping axis and group size
 * (codec PR review by 0z5a: put format/axis/group_size in the descriptor). */
typedef struct kvq_stream {
  uint32_t version;          /* KVQ_FORMAT_VERSION */
  uint8_t bits;              /* 4 */
  uint8_t kind;              /* KVQ_K (groups over rows) or KVQ_V (groups over channels) */
  uint16_t group;            /* 64 */
  uint8_t nibble_order;      /* KVQ_NIBBLE_LO_FIRST */
  uint8_t kgroup;            /* KVQ_KGROUP_COMPACT or KVQ_KGROUP_TILE (K streams; V ignores it) */
  uint8_t format;            /* KVQ_FMT_INT4 (group 64) or KVQ_FMT_NVFP4 (group 16) */
  uint8_t reserved;
  int32_t n_rows;            /* stored rows: n_tokens if dense, |active set| if sparse */
  int32_t n_tokens;          /* logical tokens T of the request */
  int32_t n_heads;           /* KV heads H */
  int32_t head_dim;          /* channels D */
  uint8_t* codes;
  uint16_t* mins;
  uint16_t* scales;
  const int32_t* active_idx; /* NULL: dense */
  int32_t* tile_dir;         /* sparse streams: written by kvq_encode_residual, read by attention/reconstruct */
  int32_t row_cap;           /* rows per head the planes hold (>= n_rows; 0: n_rows) */
  int32_t token_cap;         /* tokens the K groups, index and tile directory hold (>= n_tokens; 0: n_tokens) */
} kvq_stream;

/* Fill the format fields of `s` and clear its pointers. */
kvq_status kvq_stream_init(kvq_stream* s, int kind, int n_rows, int n_tokens, int n_heads, int head_dim);

/* Set the element format of `s` (KVQ_FMT_INT4 or KVQ_FMT_NVFP4) and its group
 * size (64 or 16). Call before kvq_plane_bytes. */
kvq_status kvq_stream_set_format(kvq_stream* s, int format);

/* Give the planes of `s` room to grow (kvq_append_tile): row_cap rows per head
 * and token_cap tokens. Every plane is then laid out with the capacities in
 * place of the counts (codes [H][row_cap][D/2], V params [H][row_cap][..], K
 * params [H][groups of the capacity][D], index [row_cap], tile directory
 * [ceil(token_cap/64)+1]); readers index by the capacities and read the first
 * n_rows / n_tokens. Call before kvq_plane_bytes. */
kvq_status kvq_stream_set_capacity(kvq_stream* s, int row_cap, int token_cap);

/* Bytes to allocate for one plane of `s` (KVQ_PLANE_*), rounded up to 16. The
 * index plane is at least 16 bytes, so that an empty sparse set still has a
 * non-NULL active_idx (NULL marks a dense stream). */
size_t kvq_plane_bytes(const kvq_stream* s, int plane);

/* Byte-exact storage of one stream: codes + FP16 mins and scales (+ 4 bytes per
 * row of sparse index), without the 16-byte allocation rounding and without the
 * derived tile directory. 4.5 bits per element on full groups (codec PR review
 * by 0z5a); partial groups pay their padding (RFC §7.4). */
int64_t kvq_stream_payload_bytes(int kind, int n_rows, int n_heads, int head_dim, int sparse);
/* The same for any K grouping and format: a tile-grouped sparse K stream
 * stores ceil(n_tokens/64) groups per (head, channel) whatever n_rows is; an
 * NVFP4 stream stores its codes, one E4M3 byte per 16 channels of a stored row
 * and head, and the 4-byte FP32 tensor scale (4.5 bits per element + 4 bytes). */
int64_t kvq_stream_payload_bytes_ex(int kind, int n_rows, int n_tokens, int n_heads, int head_dim, int sparse,
                                    int kgroup, int format);

/*
 * Encode the loop-1 base of K or V (RFC §3.3: X̂[1] = deq(q(X[1]))).
 *   x    BF16 [n_tokens][n_heads][head_dim], logical token-major, device.
 *   out  dense stream (n_rows == n_tokens, active_idx NULL) whose codes, mins
 *        and scales planes are written.
 */
kvq_status kvq_encode_base(const uint16_t* x, const kvq_stream* out, kvq_cuda_stream stream);

/*
 * Encode the residual of loop r = n_prev + 1 (RFC §3.3: delta[r] = X[r] -
 * X̂[r-1], subtracting the reconstructed predecessor, which the kernel rebuilds
 * from the packed chain at each stored row).
 *   x_r   BF16 [n_tokens][n_heads][head_dim] source of loop r, logical order.
 *   prev  n_prev descriptors of loops 1..r-1 (prev[0] the dense base); sparse
 *         ones must carry their tile_dir.
 *   out   stream of loop r: dense (active_idx NULL) or compact sparse over the
 *         ascending active rows in out->active_idx (RFC §3.3: only active tokens
 *         store a residual; K groups then run over compact rows, codec PR review
 *         by 0z5a). For a sparse `out`, out->tile_dir must point to
 *         kvq_plane_bytes(out, KVQ_PLANE_TILE_DIR) bytes and is written too.
 * Preconditions (not checked on the device): active_idx ascending without
 * duplicates, inside [0, n_tokens); nested in the previous sparse loop's set
 * (RFC §3.1). Values |x| <= 65504 so FP16 metadata stays finite.
 */
kvq_status kvq_encode_residual(const uint16_t* x_r, const kvq_stream* prev, int n_prev, const kvq_stream* out,
                               kvq_cuda_stream stream);

/* Build tile_dir[0..ceil(n_tokens/64)] for an ascending active index list:
 * tile_dir[k] = count of indices < 64k (the compact row where logical tile k
 * starts; RFC §3.3 explicit logical-to-compact maps). */
kvq_status kvq_build_tile_dir(const int32_t* active_idx, int n_rows, int n_tokens, int32_t* tile_dir,
                              kvq_cuda_stream stream);

/*
 * Append one 64-token tile to a K or V chain in place: the flush of the rolling
 * BF16 tail into the packed form in whole 64-token groups (RFC §3.3).
 *   loops[0..n_loops-1]  the chain; host descriptors, updated on success
 *          (n_tokens += 64; n_rows += the tile's stored rows of each loop).
 *          Requirements: every loop INT4; n_tokens a multiple of 64; room for
 *          the tile in the capacities (kvq_stream_set_capacity); a sparse K
 *          loop in tile grouping (KVQ_KGROUP_TILE: its new rows form a group of
 *          their own, where compact grouping would merge them into an old one).
 *   x_tile       host array [n_loops] of device pointers: BF16 [64][H][D], the
 *                tile's source of each loop.
 *   tile_active  host array [n_loops] of device pointers: a sparse loop's
 *                ascending positions (0..63) of the tile's tokens it stores,
 *                nested in the previous sparse loop's; NULL for a dense loop.
 *   n_tile_active host array [n_loops]: their counts (a dense loop: 64).
 *   workspace    >= kvq_append_workspace_bytes(n_loops) bytes of device memory,
 *                16-byte aligned.
 * The sparse loops' index and tile directory planes are extended too (K and V
 * of a request share them; appending both kinds writes the same values twice).
 * The planes then hold exactly the bytes an encode of the whole extended chain
 * would write. NVFP4 loops are refused (UNSUPPORTED): their tensor scale spans
 * the whole stream.
 */
size_t kvq_append_workspace_bytes(int n_loops);
kvq_status kvq_append_tile(kvq_stream* loops, int n_loops, const uint16_t* const* x_tile,
                           const int32_t* const* tile_active, const int* n_tile_active, void* workspace,
                           size_t workspace_bytes, kvq_cuda_stream stream);

/*
 * Reconstruct X̂ at `depth` (1 = base only) into BF16 [n_tokens][n_heads][head_dim]
 * (RFC §3.3: unpack, dequantise and sum the chain in BF16; absent tokens
 * inherit). loops[0..depth-1] describe loops 1..depth of one K or V chain.
 */
kvq_status kvq_reconstruct(const kvq_stream* loops, int depth, uint16_t* out, kvq_cuda_stream stream);

/* Per-request reference to the packed K and V chains (one entry per loop),
 * read by the attention kernel and by the batched codec calls from DEVICE
 * memory (an array of kvq_request, one per request). The batched encode
 * writes the planes (and, for a sparse loop, the tile_dir) of the loop it
 * encodes; every other call only reads through these pointers. */
#define KVQ_LOOP_K_TILE 1  /* kvq_loop_ref.flags: the K planes use KVQ_KGROUP_TILE */
#define KVQ_LOOP_K_NVFP4 2 /* kvq_loop_ref.flags: the K planes are NVFP4 */
#define KVQ_LOOP_V_NVFP4 4 /* kvq_loop_ref.flags: the V planes are NVFP4 */

typedef struct kvq_loop_ref {
  int32_t n_rows;
  int32_t flags;             /* KVQ_LOOP_* bits */
  const int32_t* active_idx; /* NULL: dense */
  int32_t* tile_dir;         /* required for sparse loops */
  uint8_t* k_codes;
  uint16_t* k_mins;
  uint16_t* k_scales;
  uint8_t* v_codes;
  uint16_t* v_mins;
  uint16_t* v_scales;
  int32_t row_cap;           /* rows per head of the planes (0: n_rows) */
  int32_t kgroup_cap;        /* K groups per head of the K param planes (0: those of n_rows) */
} kvq_loop_ref;

/*
 * BF16 segments read by the decode attention next to the packed chain (RFC
 * §3.3: a rolling BF16 tail of the newest tokens, flushed into the packed form
 * in whole 64-token groups, so 64..127 tokens remain; INT4 codec PR review:
 * the first tokens and a recent window kept in BF16).
 *   sink: the first n_sink tokens (n_sink <= n_tokens) are read from sink_k /
 *         sink_v (BF16 [n_sink][H][D]) instead of the packed chain;
 *   tail: n_tail further tokens (positions n_tokens .. n_tokens + n_tail - 1)
 *         from tail_k / tail_v (BF16 [n_tail][H][D]).
 * Zero counts (the default of kvq_request_fill) read the packed chain alone.
 * Pointers must be 16-byte aligned when their count is nonzero; a request
 * whose segment fields are inconsistent gets a NaN output and sets the error
 * word, like any inconsistent table entry.
 */
#define KVQ_MAX_SEGMENT 1024 /* largest n_sink + n_tail per request */

typedef struct kvq_request {
  int32_t n_tokens; /* T of this request (>= 0) */
  int32_t n_loops;  /* loops stored (>= the requested depth) */
  kvq_loop_ref loop[KVQ_MAX_LOOPS];
  int32_t n_sink;   /* BF16 sink tokens (0: none) */
  int32_t n_tail;   /* BF16 tail tokens (0: none) */
  const uint16_t* sink_k;
  const uint16_t* sink_v;
  const uint16_t* tail_k;
  const uint16_t* tail_v;
} kvq_request;

/* Host helper: fill one kvq_request from the K and V stream descriptors of a
 * request (n_loops of each). Checks that K and V agree on rows and sets. */
kvq_status kvq_request_fill(const kvq_stream* k_loops, const kvq_stream* v_loops, int n_loops, kvq_request* out);

/*
 * Batched tail flush: one 64-token tile appended to the K and V chains of every
 * request of a DEVICE table, all loops in one call (same bytes as
 * kvq_append_tile per request).
 *   reqs    DEVICE table (kvq_request_fill entries of growable streams); updated in
 *           place: n_tokens += 64 and each loop's n_rows += its tile rows. Each
 *           request: n_loops loops (1..4), whole tiles so far, INT4 loops with
 *           room for the tile (row_cap, kgroup_cap), sparse loops in tile grouping.
 *           A request that does not qualify is left unchanged and sets bit 1 of the
 *           error word.
 *   xk_tile, xv_tile  DEVICE arrays [n_loops * n_requests] (loop-major) of device
 *           pointers to the tile's BF16 [64][H][D] sources.
 *   tile_active  DEVICE array [n_loops * n_requests] of device pointers to a sparse
 *           loop's ascending positions 0..63 (NULL for a dense loop);
 *           n_tile_active DEVICE int32 [n_loops * n_requests], their counts (64 dense).
 *   workspace  >= kvq_append_batch_workspace_bytes(n_requests), 16-byte aligned;
 *           int32 error word at offset 0 (bit 1 refused request, bit 4 bad positions).
 */
size_t kvq_append_batch_workspace_bytes(int n_requests);
kvq_status kvq_append_tile_batch(kvq_request* reqs, int n_requests, int n_heads, int head_dim, int n_loops,
                                 const uint16_t* const* xk_tile, const uint16_t* const* xv_tile,
                                 const int32_t* const* tile_active, const int32_t* n_tile_active, void* workspace,
                                 size_t workspace_bytes, kvq_cuda_stream stream);

/* Workspace bytes the batched codec calls need for n_requests requests. */
size_t kvq_batch_workspace_bytes(int n_requests);

/*
 * Batched encode of loop `loop` (0 = the loop-1 base) of K or V (`kind`) for
 * n_requests requests, same arithmetic as kvq_encode_base / kvq_encode_residual.
 *   reqs  DEVICE table [n_requests]: loops 0..loop-1 are read as the
 *         predecessor chain; loop `loop` gives the rows to store (dense, or
 *         sparse with its active_idx) and the planes written. For a sparse
 *         loop its tile_dir is written as well (both kinds write the same
 *         values; K and V of one request share the active set).
 *   x     DEVICE array [n_requests] of device pointers to BF16 [T_b][H][D]
 *         sources of this loop.
 *   workspace  >= kvq_batch_workspace_bytes(n_requests) bytes, 16-byte aligned.
 * Table contents are preconditions (as for the single-request calls); an
 * inconsistent sparse tile map sets bit 4 of the int32 error word at offset 0
 * of the workspace. Every loop of the chain must be INT4 (see the _ex form).
 */
kvq_status kvq_encode_batch(const kvq_request* reqs, int n_requests, int n_heads, int head_dim, int kind, int loop,
                            const uint16_t* const* x, void* workspace, size_t workspace_bytes,
                            kvq_cuda_stream stream);

/* kvq_encode_batch for chains with NVFP4 residual loops: bit j of nvfp4_loops
 * says that loop j of `kind` is NVFP4 in every request of the table (bit 0,
 * the base, must be clear). A request whose loop flags disagree with the mask
 * is skipped and sets bit 64 of the error word. */
kvq_status kvq_encode_batch_ex(const kvq_request* reqs, int n_requests, int n_heads, int head_dim, int kind,
                               int loop, const uint16_t* const* x, uint32_t nvfp4_loops, void* workspace,
                               size_t workspace_bytes, kvq_cuda_stream stream);

/* Batched reconstruction at `depth` of K or V for n_requests requests into
 * out[b] (DEVICE array of device pointers to BF16 [T_b][H][D]). */
kvq_status kvq_reconstruct_batch(const kvq_request* reqs, int n_requests, int n_heads, int head_dim, int kind,
                                 int depth, uint16_t* const* out, void* workspace, size_t workspace_bytes,
                                 kvq_cuda_stream stream);

/* kvq_reconstruct_batch for chains with NVFP4 residual loops (nvfp4_loops as
 * in kvq_encode_batch_ex). */
kvq_status kvq_reconstruct_batch_ex(const kvq_request* reqs, int n_requests, int n_heads, int head_dim, int kind,
                                    int depth, uint16_t* const* out, uint32_t nvfp4_loops, void* workspace,
                                    size_t workspace_bytes, kvq_cuda_stream stream);

/* Workspace bytes kvq_decode_attn_packed needs on the current device. */
size_t kvq_decode_attn_workspace_bytes(int n_requests, int n_heads, int n_q_heads, int head_dim);

#define KVQ_ATTN_AUTO 0 /* tensor-core kernel for depth <= 4, CUDA-core kernel beyond */
#define KVQ_ATTN_SIMT 1 /* CUDA-core kernel: FP32 decode of the chain per element, FP32 dot products */
#define KVQ_ATTN_MMA 2  /* tensor-core kernel (depth <= 4): INT4 tables run the subnormal-code kernel (Q' and the
                           K-min terms built once per tile). With KVQ_ATTN_NVFP4 both that kernel and the general
                           one are launched and the plan kernel picks one: a call in which some request holds an
                           NVFP4 loop within depth runs the general kernel, any other call the subnormal-code one
                           (the other launch leaves at once) */
#define KVQ_ATTN_MMA_GENERAL 3 /* the general tensor-core kernel (depth <= 4) for every table: codes as FP16 64 + c,
                                 Q' rebuilt per warp; the form that reads NVFP4 loops */
#define KVQ_ATTN_TCGEN05 4 /* INT4 tables on the tcgen05 form of the subnormal-code kernel (codes in tensor memory and
                             shared memory, accumulators in tensor memory, warp-specialised, one block per SM; slower
                             than KVQ_ATTN_MMA on decode shapes); NVFP4 tables as KVQ_ATTN_MMA */
#define KVQ_ATTN_NVFP4 8 /* OR-ed into algo: the table may hold NVFP4 residual loops (an INT4 table
                           passed with it costs one extra, empty kernel launch). Without it the
                           tensor-core kernel refuses such a request (NaN output, error bit 64); the
                           CUDA-core kernel reads either format. kvq_decode_attn_packed and the
                           no-alloc entry run without it (INT4 tables). */

/*
 * Packed-KV GQA decode attention at `depth` (RFC §3.2: historical K/V are read
 * at the requested depth and reconstructed if compressed; §3.3: readers consume
 * packed base/residual tiles directly, with no BF16 shadow cache).
 *   reqs       DEVICE array [n_requests] of kvq_request.
 *   q          BF16 [n_requests][n_q_heads][head_dim], one decode query per request.
 *   out        FP32 [n_requests][n_q_heads][head_dim].
 *   softmax_scale  usually 1/sqrt(head_dim) (RFC §3.2).
 *   workspace  DEVICE scratch of >= kvq_decode_attn_workspace_bytes(...) bytes,
 *              16-byte aligned; int32 at offset 0 is an error word the kernels
 *              set (nonzero) when a request's table entry is inconsistent; that
 *              request's output is then NaN.
 * Query head hq reads KV head hq / (n_q_heads / n_heads). Softmax and all
 * accumulation are FP32. A request with n_tokens == 0 gets a zero output.
 */
kvq_status kvq_decode_attn_packed(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads,
                                  int head_dim, int depth, const uint16_t* q, float softmax_scale, float* out,
                                  void* workspace, size_t workspace_bytes, kvq_cuda_stream stream);

/* Same, choosing the kernel (KVQ_ATTN_*). */
kvq_status kvq_decode_attn_packed_ex(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads,
                                     int head_dim, int depth, const uint16_t* q, float softmax_scale, float* out,
                                     void* workspace, size_t workspace_bytes, int algo, kvq_cuda_stream stream);

/*
 * Sparse decode attention over the packed chains (RFC §3.2). At the reference
 * loop the full attention is computed and, per query head, the n_select keys
 * of largest probability are kept (equal probabilities: lower position
 * first) with their probability mass m, the full output O_ref and their
 * contribution C_ref = sum over S of p_t v_t; a later loop r reads only the
 * keys of S at its own depth and returns
 *     O = O_ref - C_ref + m * softmax(q_r K_r[S]^T * scale) V_r[S].
 * K = min(n_select, n_tokens) keys per (request, query head). All of it is
 * FP32 on the FP32 decode of the packed chain. Requests with BF16 segments
 * (n_sink or n_tail nonzero) and requests longer than max_tokens are refused
 * on the device: their outputs are NaN and bit 1 of the error word is set.
 */
size_t kvq_sparse_workspace_bytes(int n_requests, int n_heads, int n_q_heads, int head_dim, int max_tokens);

/* Reference loop at ref_depth (usually 2).
 *   q_ref     BF16 [n_requests][n_q_heads][head_dim].
 *   sel_idx   int32 [n_requests][n_q_heads][n_select]: the selected positions in
 *             ascending order, -1 past the request's K.
 *   mass      FP32 [n_requests][n_q_heads]; o_ref, c_ref FP32 [..][..][head_dim]
 *             (16-byte aligned).
 *   workspace >= kvq_sparse_workspace_bytes(...) bytes, 16-byte aligned; int32 at
 *             offset 0 is the error word (bits: 1 inconsistent request, ...). */
kvq_status kvq_sparse_ref_state(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads, int head_dim,
                                int ref_depth, const uint16_t* q_ref, float softmax_scale, int n_select,
                                int max_tokens, int32_t* sel_idx, float* mass, float* o_ref, float* c_ref,
                                void* workspace, size_t workspace_bytes, kvq_cuda_stream stream);

/* A later loop at `depth` with the state of kvq_sparse_ref_state (same n_select
 * and max_tokens); out FP32 [n_requests][n_q_heads][head_dim]. workspace: at
 * least 16 bytes, 16-byte aligned; int32 at offset 0 is the error word (bit 32:
 * a selected position outside its request, which is then left out).
 * Two kernels compute the later loop:
 *   - with a workspace of at least kvq_sparse_decode_workspace_bytes(...), a
 *     depth <= 4, 1, 2, 4 or 8 query heads per KV head and a 16-byte aligned
 *     out, the selections become a key mask per (request, query head) and the
 *     packed tensor-core attention (kvq_decode_attn_packed) attends with the
 *     unselected keys' logits dropped; a small kernel then applies the
 *     correction;
 *   - otherwise, or when the selection is small (n_select * 64 <= max_tokens:
 *     the key-masked attention still reads every tile, while gathering so few
 *     keys one by one reads far fewer bytes), a kernel that gathers the
 *     selected keys one by one.
 * kvq_sparse_decode_attn reads NVFP4 loops (it passes KVQ_ATTN_NVFP4). */
kvq_status kvq_sparse_decode_attn(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads, int head_dim,
                                  int depth, const uint16_t* q, float softmax_scale, int n_select, int max_tokens,
                                  const int32_t* sel_idx, const float* mass, const float* o_ref, const float* c_ref,
                                  float* out, void* workspace, size_t workspace_bytes, kvq_cuda_stream stream);

/* Workspace bytes with which kvq_sparse_decode_attn takes the tensor-core path:
 * the packed attention's workspace (kvq_decode_attn_workspace_bytes, rounded up
 * to 256 bytes) followed by the key masks, 2 * ceil(max_tokens / 64) uint32
 * words per (request, query head). 0 for invalid sizes. */
size_t kvq_sparse_decode_workspace_bytes(int n_requests, int n_heads, int n_q_heads, int head_dim, int max_tokens);

/* Same as kvq_sparse_decode_attn, choosing the kernel: algo KVQ_ATTN_AUTO (the
 * choice above), KVQ_ATTN_SIMT (the per-key
 * kernel) or KVQ_ATTN_MMA (the tensor-core path, or KVQ_ERR_UNSUPPORTED /
 * KVQ_ERR_WORKSPACE when it cannot run), ORed with KVQ_ATTN_NVFP4 when the table
 * may hold NVFP4 loops. Without that flag the tensor-core path refuses requests
 * with NVFP4 loops (NaN output, bit 64 of the error word), as
 * kvq_decode_attn_packed_ex does. */
kvq_status kvq_sparse_decode_attn_ex(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads, int head_dim,
                                     int depth, const uint16_t* q, float softmax_scale, int n_select, int max_tokens,
                                     const int32_t* sel_idx, const float* mass, const float* o_ref, const float* c_ref,
                                     float* out, void* workspace, size_t workspace_bytes, int algo,
                                     kvq_cuda_stream stream);

/* Bytes of the static device scratch used by kvq_decode_attn_packed_noalloc. */
#define KVQ_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * Packed-KV decode attention that allocates nothing and takes no workspace.
 * There is no counterpart on the pages: it serves callers that cannot
 * allocate device memory (code running under CUDA graph capture, plugins in a
 * serving process that owns all device allocations, hosts whose allocator the
 * library cannot reach). Arguments and results are those of
 * kvq_decode_attn_packed (an INT4 table: a request holding NVFP4 loops is
 * refused, as kvq_decode_attn_packed_ex refuses it without KVQ_ATTN_NVFP4).
 * Host-side checks return the same status codes. The device-side error word
 * lives in the static scratch, which the caller cannot read: a request the
 * kernels refuse (NVFP4 loops, an inconsistent table entry, a timed-out
 * pipeline wait) is seen only as NaN in its output rows. The scratch it needs
 * lives in a file-scope device array of KVQ_NOALLOC_SCRATCH_BYTES (32 MiB),
 * reserved on every device that loads it until the process exits.
 *   - Sizes whose kvq_decode_attn_workspace_bytes() exceed 32 MiB are rejected
 *     with KVQ_ERR_WORKSPACE before any launch (on a 152-SM GB300 that is about
 *     6800 request x KV-head pairs per call).
 *   - The first call on a device looks up the array's device address with that
 *     device current; make that first call before any stream capture. The
 *     address is kept for the life of the process: do not reset the device
 *     (cudaDeviceReset) once this entry point has been used.
 *   - Every call shares the array and leaves its contents behind; calls that
 *     overlap on the GPU race on it and must be serialised by the caller.
 */
kvq_status kvq_decode_attn_packed_noalloc(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads,
                                          int head_dim, int depth, const uint16_t* q, float softmax_scale,
                                          float* out, kvq_cuda_stream stream);

/* Human-readable name of a status code. */
const char* kvq_status_string(kvq_status s);

/* One-line reason for the last failing call on this thread ("" if none). */
const char* kvq_last_error(void);

/* Library and format version: (major << 16) | minor. */
uint32_t kvq_version(void);

/* Number of CUDA kernels this library has launched in the calling process
 * (host-side counter; for accounting launches in timed regions). */
uint64_t kvq_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H_ */
