// kvq_api.cu — the extern "C" entry points of libkvq.so (declared in
// include/kvq.h): host-side argument checks, then asynchronous launches on the
// caller's stream. Nothing here allocates device memory or synchronises.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "kvq_attn_common.cuh"
#include "kvq_sparse.cuh"

using namespace kvq;

namespace {

thread_local char g_err[512] = {0};

kvq_status fail(kvq_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return s;
}

kvq_status ok() {
  g_err[0] = 0;
  return KVQ_OK;
}

kvq_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t round16(size_t x) { return (x + 15) / 16 * 16; }

// Checks the format fields of a descriptor (not its pointers).
kvq_status check_format(const kvq_stream* s, const char* name) {
  if (s == nullptr) return fail(KVQ_ERR_BAD_ARG, "%s is NULL", name);
  if (s->version != KVQ_FORMAT_VERSION) return fail(KVQ_ERR_UNSUPPORTED, "%s: format version %u", name, s->version);
  const bool fmt_ok = (s->format == KVQ_FMT_INT4 && s->group == KVQ_GROUP) ||
                      (s->format == KVQ_FMT_NVFP4 && s->group == 16);
  if (s->bits != KVQ_BITS || !fmt_ok || s->nibble_order != KVQ_NIBBLE_LO_FIRST)
    return fail(KVQ_ERR_UNSUPPORTED, "%s: bits %d format %d group %d nibble order %d", name, s->bits, s->format,
                s->group, s->nibble_order);
  if (s->kind != KVQ_K && s->kind != KVQ_V) return fail(KVQ_ERR_BAD_ARG, "%s: kind %d", name, s->kind);
  if (s->kgroup != KVQ_KGROUP_COMPACT && s->kgroup != KVQ_KGROUP_TILE)
    return fail(KVQ_ERR_UNSUPPORTED, "%s: K grouping %d", name, s->kgroup);
  if (s->n_tokens < 0 || s->n_rows < 0 || s->n_rows > s->n_tokens)
    return fail(KVQ_ERR_BAD_ARG, "%s: n_rows %d n_tokens %d", name, s->n_rows, s->n_tokens);
  if (s->n_heads < 1 || s->n_heads > 1024) return fail(KVQ_ERR_BAD_ARG, "%s: n_heads %d", name, s->n_heads);
  if (s->head_dim != kD) return fail(KVQ_ERR_UNSUPPORTED, "%s: head_dim %d (kernels support 128)", name, s->head_dim);
  if (s->active_idx == nullptr && s->n_rows != s->n_tokens)
    return fail(KVQ_ERR_BAD_ARG, "%s: dense stream with n_rows %d != n_tokens %d", name, s->n_rows, s->n_tokens);
  if (s->row_cap < 0 || (s->row_cap > 0 && s->row_cap < s->n_rows) || s->token_cap < 0 ||
      (s->token_cap > 0 && s->token_cap < s->n_tokens) || (s->row_cap > 0) != (s->token_cap > 0))
    return fail(KVQ_ERR_BAD_ARG, "%s: capacities row %d token %d for n_rows %d n_tokens %d", name, s->row_cap,
                s->token_cap, s->n_rows, s->n_tokens);
  return KVQ_OK;
}

// Rows per head and tokens the planes of s are laid out for.
int row_capacity(const kvq_stream* s) { return s->row_cap > 0 ? s->row_cap : s->n_rows; }
int token_capacity(const kvq_stream* s) { return s->token_cap > 0 ? s->token_cap : s->n_tokens; }

// Checks pointers of a stream that is read (need_dir: sparse streams must carry tile_dir).
kvq_status check_planes(const kvq_stream* s, const char* name, bool need_dir) {
  kvq_status st = check_format(s, name);
  if (st != KVQ_OK) return st;
  if (s->n_rows == 0) return KVQ_OK;
  if (!s->codes || !s->mins || !s->scales) return fail(KVQ_ERR_BAD_ARG, "%s: NULL plane", name);
  if (!aligned16(s->codes) || !aligned16(s->mins) || !aligned16(s->scales) ||
      (s->active_idx && !aligned16(s->active_idx)))
    return fail(KVQ_ERR_MISALIGNED, "%s: planes must be 16-byte aligned", name);
  if (need_dir && s->active_idx && !s->tile_dir) return fail(KVQ_ERR_BAD_ARG, "%s: sparse stream without tile_dir", name);
  return KVQ_OK;
}

bool k_tile(const kvq_stream* s) { return s->kind == KVQ_K && s->kgroup == KVQ_KGROUP_TILE; }
bool nvfp4(const kvq_stream* s) { return s->format == KVQ_FMT_NVFP4; }

// Loop-ref flag bits of a stream (K or V planes).
int32_t loop_flags(const kvq_stream* s) {
  int32_t f = k_tile(s) ? KVQ_LOOP_K_TILE : 0;
  if (nvfp4(s)) f |= s->kind == KVQ_K ? KVQ_LOOP_K_NVFP4 : KVQ_LOOP_V_NVFP4;
  return f;
}

// Bit j: loop j of the streams is NVFP4.
uint32_t nvfp4_mask(const kvq_stream* loops, int n) {
  uint32_t m = 0;
  for (int j = 0; j < n; ++j)
    if (nvfp4(&loops[j])) m |= 1u << j;
  return m;
}

void to_planes(const kvq_stream* s, LoopPlanes* p) {
  p->n_rows = s->n_rows;
  p->sparse = s->active_idx != nullptr;
  p->ktile = k_tile(s);
  p->kgroups = k_groups_of(k_tile(s), row_capacity(s), token_capacity(s));
  p->stride = row_capacity(s);
  p->fmt = s->format;
  p->active = s->active_idx;
  p->tile_dir = s->tile_dir;
  p->codes = s->codes;
  p->mins = s->mins;
  p->scales = s->scales;
}

kvq_status build_chain(const kvq_stream* loops, int depth, Chain* C, const char* name) {
  if (depth < 1 || depth > KVQ_MAX_LOOPS) return fail(KVQ_ERR_BAD_ARG, "%s: depth %d", name, depth);
  if (loops == nullptr) return fail(KVQ_ERR_BAD_ARG, "%s is NULL", name);
  for (int j = 0; j < depth; ++j) {
    char nm[64];
    snprintf(nm, sizeof nm, "%s[%d]", name, j);
    kvq_status st = check_planes(&loops[j], nm, true);
    if (st != KVQ_OK) return st;
    if (loops[j].kind != loops[0].kind || loops[j].n_tokens != loops[0].n_tokens ||
        loops[j].n_heads != loops[0].n_heads)
      return fail(KVQ_ERR_BAD_ARG, "%s: loops disagree on kind, n_tokens or n_heads", name);
  }
  if (loops[0].active_idx != nullptr) return fail(KVQ_ERR_BAD_ARG, "%s[0]: the base must be dense", name);
  if (nvfp4(&loops[0])) return fail(KVQ_ERR_UNSUPPORTED, "%s[0]: the base must be INT4", name);
  memset(C, 0, sizeof *C);
  C->depth = depth;
  C->kind = loops[0].kind;
  C->n_tokens = loops[0].n_tokens;
  C->n_heads = loops[0].n_heads;
  for (int j = 0; j < depth; ++j) to_planes(&loops[j], &C->loop[j]);
  return KVQ_OK;
}

int sm_count(int device) {
  static int cache[64] = {0};
  if (device < 0 || device >= 64) return 0;
  if (cache[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
    cache[device] = n;
  }
  return cache[device];
}

constexpr int kMaxCtasPerSm = 8;

}  // namespace

namespace kvq {
void set_error_message(const char* msg) { snprintf(g_err, sizeof g_err, "%s", msg); }

static std::atomic<unsigned long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int attn_ctas(int algo, int device) {
  int sms = sm_count(device);
  if (sms <= 0) return 0;
  // the tensor-core kernel runs two independent groups (virtual CTAs) per block
  int per_sm = (algo == KVQ_ATTN_SIMT) ? 4 : 2;
  if (per_sm > kMaxCtasPerSm) per_sm = kMaxCtasPerSm;
  return sms * per_sm;
}
}  // namespace kvq

extern "C" {

uint32_t kvq_version(void) { return (1u << 16) | KVQ_FORMAT_VERSION; }

uint64_t kvq_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_BAD_ARG: return "KVQ_ERR_BAD_ARG";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED";
    case KVQ_ERR_MISALIGNED: return "KVQ_ERR_MISALIGNED";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA";
    default: return "KVQ_ERR_UNKNOWN";
  }
}

const char* kvq_last_error(void) { return g_err; }

kvq_status kvq_stream_init(kvq_stream* s, int kind, int n_rows, int n_tokens, int n_heads, int head_dim) {
  if (s == nullptr) return fail(KVQ_ERR_BAD_ARG, "stream is NULL");
  memset(s, 0, sizeof *s);
  s->version = KVQ_FORMAT_VERSION;
  s->bits = KVQ_BITS;
  s->kind = uint8_t(kind);
  s->group = KVQ_GROUP;
  s->nibble_order = KVQ_NIBBLE_LO_FIRST;
  s->n_rows = n_rows;
  s->n_tokens = n_tokens;
  s->n_heads = n_heads;
  s->head_dim = head_dim;
  s->format = KVQ_FMT_INT4;
  if (kind != KVQ_K && kind != KVQ_V) return fail(KVQ_ERR_BAD_ARG, "kind %d", kind);
  if (n_tokens < 0 || n_rows < 0 || n_rows > n_tokens || n_heads < 1 || head_dim < 2 || (head_dim & 1))
    return fail(KVQ_ERR_BAD_ARG, "sizes n_rows %d n_tokens %d n_heads %d head_dim %d", n_rows, n_tokens, n_heads,
                head_dim);
  return ok();
}

kvq_status kvq_stream_set_capacity(kvq_stream* s, int row_cap, int token_cap) {
  if (s == nullptr) return fail(KVQ_ERR_BAD_ARG, "stream is NULL");
  if (row_cap < s->n_rows || token_cap < s->n_tokens || row_cap > token_cap)
    return fail(KVQ_ERR_BAD_ARG, "capacities row %d token %d below n_rows %d n_tokens %d (or rows above tokens)",
                row_cap, token_cap, s->n_rows, s->n_tokens);
  s->row_cap = row_cap;
  s->token_cap = token_cap;
  return ok();
}

kvq_status kvq_stream_set_format(kvq_stream* s, int format) {
  if (s == nullptr) return fail(KVQ_ERR_BAD_ARG, "stream is NULL");
  if (format == KVQ_FMT_INT4) {
    s->format = KVQ_FMT_INT4;
    s->group = KVQ_GROUP;
  } else if (format == KVQ_FMT_NVFP4) {
    if (s->head_dim % 16 != 0) return fail(KVQ_ERR_UNSUPPORTED, "NVFP4 needs head_dim %% 16 == 0");
    s->format = KVQ_FMT_NVFP4;
    s->group = 16;
  } else {
    return fail(KVQ_ERR_BAD_ARG, "format %d", format);
  }
  return ok();
}

size_t kvq_plane_bytes(const kvq_stream* s, int plane) {
  if (s == nullptr) return 0;
  const int64_t n = s->n_rows, H = s->n_heads, D = s->head_dim;
  const int64_t nc = row_capacity(s), tc = token_capacity(s);
  if (nvfp4(s) && plane == KVQ_PLANE_MINS) return round16(size_t(H * nc * (D / 16)));  // E4M3 block scales
  if (nvfp4(s) && plane == KVQ_PLANE_SCALES) return 16;                              // FP32 tensor-scale record
  switch (plane) {
    case KVQ_PLANE_CODES: return round16(size_t(H * nc * (D / 2)));
    case KVQ_PLANE_MINS:
    case KVQ_PLANE_SCALES:
      if (s->kind == KVQ_K) return round16(size_t(2 * H * k_groups_of(k_tile(s), int(nc), int(tc)) * D));
      return round16(size_t(2 * H * nc * cdiv(D, KVQ_GROUP)));
    case KVQ_PLANE_INDEX: return nc > 0 ? round16(size_t(4 * nc)) : 16;  // never NULL: NULL means dense
    case KVQ_PLANE_TILE_DIR: return round16(size_t(4 * (cdiv(tc, KVQ_TILE) + 1)));
    default: return 0;
  }
}

int64_t kvq_stream_payload_bytes_ex(int kind, int n_rows, int n_tokens, int n_heads, int head_dim, int sparse,
                                    int kgroup, int format) {
  const int64_t n = n_rows, H = n_heads, D = head_dim;
  if (format == KVQ_FMT_NVFP4) return n > 0 ? H * n * (D / 2) + H * n * (D / 16) + 4 + (sparse ? 4 * n : 0) : 0;
  const bool tile = kgroup == KVQ_KGROUP_TILE && sparse;
  int64_t params = (kind == KVQ_K) ? H * k_groups_of(tile, n_rows, n_tokens) * D : H * n * cdiv(D, KVQ_GROUP);
  return H * n * (D / 2) + 2 * 2 * params + (sparse ? 4 * n : 0);
}

int64_t kvq_stream_payload_bytes(int kind, int n_rows, int n_heads, int head_dim, int sparse) {
  return kvq_stream_payload_bytes_ex(kind, n_rows, n_rows, n_heads, head_dim, sparse, KVQ_KGROUP_COMPACT,
                                     KVQ_FMT_INT4);
}

// Planes of a stream descriptor as one loop entry of a request.
static void to_loop_ref(const kvq_stream* s, kvq_loop_ref* L) {
  L->n_rows = s->n_rows;
  L->flags |= loop_flags(s);
  if (s->row_cap > 0) {
    L->row_cap = s->row_cap;
    if (s->kind == KVQ_K) L->kgroup_cap = k_groups_of(k_tile(s), s->row_cap, s->token_cap);
  }
  L->active_idx = s->active_idx;
  L->tile_dir = s->tile_dir;
  if (s->kind == KVQ_K) {
    L->k_codes = s->codes;
    L->k_mins = s->mins;
    L->k_scales = s->scales;
  } else {
    L->v_codes = s->codes;
    L->v_mins = s->mins;
    L->v_scales = s->scales;
  }
}

static kvq_status current_sms(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
  *sms = sm_count(dev);
  if (*sms <= 0) return fail(KVQ_ERR_CUDA, "cannot read the SM count of device %d", dev);
  return KVQ_OK;
}

static kvq_status run_single(CodecArgs& a, int mode, cudaStream_t s, const char* what) {
  int sms = 0;
  kvq_status st = current_sms(&sms);
  if (st != KVQ_OK) return st;
  return cuda_status(launch_codec(a, mode, nullptr, sms, s), what);
}

kvq_status kvq_encode_base(const uint16_t* x, const kvq_stream* out, kvq_cuda_stream stream) {
  kvq_status st = check_planes(out, "out", false);
  if (st != KVQ_OK) return st;
  if (out->active_idx != nullptr) return fail(KVQ_ERR_BAD_ARG, "out: the base stream must be dense");
  if (nvfp4(out)) return fail(KVQ_ERR_UNSUPPORTED, "out: the base must be INT4 (NVFP4 is a residual format)");
  if (out->n_rows == 0) return ok();
  if (x == nullptr) return fail(KVQ_ERR_BAD_ARG, "x is NULL");
  if (!aligned16(x)) return fail(KVQ_ERR_MISALIGNED, "x must be 16-byte aligned");
  CodecArgs a;
  memset(&a, 0, sizeof a);
  a.H = out->n_heads;
  a.kind = out->kind;
  a.loop = 0;
  a.one.n_tokens = out->n_tokens;
  a.one.n_loops = 1;
  to_loop_ref(out, &a.one.loop[0]);
  a.one_x = x;
  return run_single(a, out->kind == KVQ_K ? kModeEncK : kModeEncV, reinterpret_cast<cudaStream_t>(stream),
                    "encode_base launch");
}

kvq_status kvq_build_tile_dir(const int32_t* active_idx, int n_rows, int n_tokens, int32_t* tile_dir,
                              kvq_cuda_stream stream) {
  if (n_rows < 0 || n_tokens < 0 || n_rows > n_tokens)
    return fail(KVQ_ERR_BAD_ARG, "n_rows %d n_tokens %d", n_rows, n_tokens);
  if (tile_dir == nullptr || active_idx == nullptr) return fail(KVQ_ERR_BAD_ARG, "NULL active_idx or tile_dir");
  CodecArgs a;
  memset(&a, 0, sizeof a);
  a.H = 1;
  a.loop = 0;
  a.one.n_tokens = n_tokens;
  a.one.n_loops = 1;
  a.one.loop[0].n_rows = n_rows;
  a.one.loop[0].active_idx = active_idx;
  a.one.loop[0].tile_dir = tile_dir;
  return run_single(a, kModeTileDir, reinterpret_cast<cudaStream_t>(stream), "tile_dir launch");
}

kvq_status kvq_encode_residual(const uint16_t* x_r, const kvq_stream* prev, int n_prev, const kvq_stream* out,
                               kvq_cuda_stream stream) {
  if (n_prev < 1 || n_prev >= KVQ_MAX_LOOPS) return fail(KVQ_ERR_BAD_ARG, "n_prev %d", n_prev);
  Chain C;
  kvq_status st = build_chain(prev, n_prev, &C, "prev");
  if (st != KVQ_OK) return st;
  st = check_planes(out, "out", false);
  if (st != KVQ_OK) return st;
  if (out->kind != prev[0].kind || out->n_tokens != prev[0].n_tokens || out->n_heads != prev[0].n_heads)
    return fail(KVQ_ERR_BAD_ARG, "out disagrees with prev on kind, n_tokens or n_heads");
  if (out->active_idx != nullptr && out->tile_dir == nullptr)
    return fail(KVQ_ERR_BAD_ARG, "out: sparse stream needs tile_dir storage");
  if (out->n_rows > 0 && x_r == nullptr) return fail(KVQ_ERR_BAD_ARG, "x_r is NULL");
  if (out->n_rows > 0 && !aligned16(x_r)) return fail(KVQ_ERR_MISALIGNED, "x_r must be 16-byte aligned");
  CodecArgs a;
  memset(&a, 0, sizeof a);
  a.H = out->n_heads;
  a.kind = out->kind;
  a.loop = n_prev;
  a.one.n_tokens = out->n_tokens;
  a.one.n_loops = n_prev + 1;
  for (int j = 0; j < n_prev; ++j) to_loop_ref(&prev[j], &a.one.loop[j]);
  to_loop_ref(out, &a.one.loop[n_prev]);
  a.one_x = x_r;
  a.nvfp4 = nvfp4_mask(prev, n_prev) | (nvfp4(out) ? 1u << n_prev : 0u);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (nvfp4(out)) {  // the tensor-scale record: s_t and the encoder's running max |delta| start at 0
    if (out->scales == nullptr || !aligned16(out->scales)) return fail(KVQ_ERR_BAD_ARG, "out: NVFP4 scale record");
    cudaError_t e = cudaMemsetAsync(out->scales, 0, 16, s);
    if (e != cudaSuccess) return cuda_status(e, "clear tensor scale");
  }
  if (out->active_idx != nullptr) {
    st = run_single(a, kModeTileDir, s, "tile_dir launch");
    if (st != KVQ_OK) return st;
  }
  return run_single(a, out->kind == KVQ_K ? kModeEncK : kModeEncV, s, "encode_residual launch");
}

constexpr size_t kAppendLoopBytes = 320;  // per loop: 64 checked positions, a 2-entry directory, padding

size_t kvq_append_workspace_bytes(int n_loops) {
  if (n_loops < 1 || n_loops > KVQ_MAX_LOOPS) return 0;
  return 16 + size_t(n_loops) * kAppendLoopBytes;
}

kvq_status kvq_append_tile(kvq_stream* loops, int n_loops, const uint16_t* const* x_tile,
                           const int32_t* const* tile_active, const int* n_tile_active, void* workspace,
                           size_t workspace_bytes, kvq_cuda_stream stream) {
  if (n_loops < 1 || n_loops > KVQ_MAX_LOOPS) return fail(KVQ_ERR_BAD_ARG, "n_loops %d", n_loops);
  if (!loops || !x_tile || !tile_active || !n_tile_active) return fail(KVQ_ERR_BAD_ARG, "NULL argument");
  Chain C;
  kvq_status st = build_chain(loops, n_loops, &C, "loops");
  if (st != KVQ_OK) return st;
  const size_t need = kvq_append_workspace_bytes(n_loops);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return fail(KVQ_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", need);
  const int T = loops[0].n_tokens, H = loops[0].n_heads, kind = loops[0].kind;
  if (T % KVQ_TILE != 0) return fail(KVQ_ERR_BAD_ARG, "n_tokens %d is not a multiple of %d", T, KVQ_TILE);
  for (int r = 0; r < n_loops; ++r) {
    const kvq_stream& L = loops[r];
    const int m = n_tile_active[r];
    if (nvfp4(&L)) return fail(KVQ_ERR_UNSUPPORTED, "loop %d: NVFP4 streams cannot grow (per-stream tensor scale)", r);
    if (L.row_cap <= 0 || L.token_cap < T + KVQ_TILE || L.n_rows + m > L.row_cap)
      return fail(KVQ_ERR_BAD_ARG, "loop %d: capacities row %d token %d cannot take the tile", r, L.row_cap,
                  L.token_cap);
    if (L.active_idx == nullptr) {
      if (tile_active[r] != nullptr || m != KVQ_TILE)
        return fail(KVQ_ERR_BAD_ARG, "loop %d: a dense loop stores all %d tokens of the tile", r, KVQ_TILE);
    } else {
      if (tile_active[r] == nullptr || m < 0 || m > KVQ_TILE)
        return fail(KVQ_ERR_BAD_ARG, "loop %d: sparse loop needs 0..%d tile positions", r, KVQ_TILE);
      if (L.kind == KVQ_K && L.kgroup != KVQ_KGROUP_TILE)
        return fail(KVQ_ERR_UNSUPPORTED, "loop %d: a sparse K loop grows only under tile grouping", r);
    }
    if (x_tile[r] == nullptr || !aligned16(x_tile[r])) return fail(KVQ_ERR_MISALIGNED, "x_tile[%d]", r);
    if (!L.codes || !L.mins || !L.scales || (L.active_idx && !L.tile_dir))
      return fail(KVQ_ERR_BAD_ARG, "loop %d: planes missing", r);
    if (!aligned16(L.codes) || !aligned16(L.mins) || !aligned16(L.scales))
      return fail(KVQ_ERR_MISALIGNED, "loop %d: planes must be 16-byte aligned", r);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int32_t* err = reinterpret_cast<int32_t*>(ws);
  cudaError_t e = cudaMemsetAsync(err, 0, 16, s);
  if (e != cudaSuccess) return cuda_status(e, "clear error word");
  AppendIndexArgs ia;
  memset(&ia, 0, sizeof ia);
  ia.n_loops = n_loops;
  ia.T = T;
  ia.err = err;
  for (int r = 0; r < n_loops; ++r) {
    int32_t* base = reinterpret_cast<int32_t*>(ws + 16 + size_t(r) * kAppendLoopBytes);
    ia.loop[r].rel = loops[r].active_idx ? tile_active[r] : nullptr;
    ia.loop[r].rel_ws = base;
    ia.loop[r].dir_ws = base + 64;
    ia.loop[r].active = const_cast<int32_t*>(loops[r].active_idx);
    ia.loop[r].tile_dir = loops[r].tile_dir;
    ia.loop[r].n_old = loops[r].n_rows;
    ia.loop[r].n_new = n_tile_active[r];
  }
  e = launch_append_index(ia, s);
  if (e != cudaSuccess) return cuda_status(e, "append index launch");
  // tile-grouped sparse K: the groups of tiles without stored rows hold +0 min and scale
  for (int r = 0; r < n_loops && kind == KVQ_K; ++r) {
    const kvq_stream& L = loops[r];
    if (L.active_idx == nullptr) continue;
    const int m = n_tile_active[r], k = T / KVQ_TILE;
    int g0 = 0, g1 = 0;  // groups to clear
    if (m == 0 && L.n_rows > 0) g0 = k, g1 = k + 1;
    if (m > 0 && L.n_rows == 0) g0 = 0, g1 = k;  // the stream's first rows: the earlier tiles are empty
    if (g1 <= g0) continue;
    const size_t pitch = size_t(k_groups_of(true, L.row_cap, L.token_cap)) * kD * 2;
    for (uint16_t* plane : {L.mins, L.scales}) {
      e = cudaMemset2DAsync(reinterpret_cast<char*>(plane) + size_t(g0) * kD * 2, pitch, 0, size_t(g1 - g0) * kD * 2,
                            H, s);
      if (e != cudaSuccess) return cuda_status(e, "clear empty tile groups");
    }
  }
  // encode loop by loop through views of the tile's rows (tokens 0..63 of x_tile)
  for (int r = 0; r < n_loops; ++r) {
    CodecArgs a;
    memset(&a, 0, sizeof a);
    a.H = H;
    a.kind = kind;
    a.loop = r;
    a.err = err;
    a.one.n_tokens = KVQ_TILE;
    a.one.n_loops = r + 1;
    for (int j = 0; j <= r; ++j) {
      const kvq_stream& L = loops[j];
      kvq_loop_ref& V = a.one.loop[j];
      const int32_t* base = reinterpret_cast<const int32_t*>(ws + 16 + size_t(j) * kAppendLoopBytes);
      V.n_rows = n_tile_active[j];
      V.flags = loop_flags(&L);
      V.row_cap = L.row_cap;
      V.kgroup_cap = kind == KVQ_K ? k_groups_of(k_tile(&L), L.row_cap, L.token_cap) : 0;
      V.active_idx = L.active_idx ? base : nullptr;
      V.tile_dir = L.active_idx ? const_cast<int32_t*>(base + 64) : nullptr;
      uint8_t* codes = L.codes + size_t(L.n_rows) * kRowBytes;  // row n_rows of head 0; heads at row_cap
      // K: the tile's group (index T/64 under either grouping of a growable loop); V: row n_rows
      const size_t poff = kind == KVQ_K ? size_t(T / KVQ_TILE) * kD : size_t(L.n_rows) * (kD / kG);
      if (kind == KVQ_K) {
        V.k_codes = codes;
        V.k_mins = L.mins + poff;
        V.k_scales = L.scales + poff;
      } else {
        V.v_codes = codes;
        V.v_mins = L.mins + poff;
        V.v_scales = L.scales + poff;
      }
    }
    a.one_x = x_tile[r];
    st = run_single(a, kind == KVQ_K ? kModeEncK : kModeEncV, s, "append encode launch");
    if (st != KVQ_OK) return st;
  }
  for (int r = 0; r < n_loops; ++r) {
    loops[r].n_rows += n_tile_active[r];
    loops[r].n_tokens += KVQ_TILE;
  }
  return ok();
}

size_t kvq_append_batch_workspace_bytes(int n_requests) {
  if (n_requests < 0) return 0;
  return 16 + round16(size_t(n_requests + 1) * 4) + round16(size_t(n_requests) * 4);
}

kvq_status kvq_append_tile_batch(kvq_request* reqs, int n_requests, int n_heads, int head_dim, int n_loops,
                                 const uint16_t* const* xk_tile, const uint16_t* const* xv_tile,
                                 const int32_t* const* tile_active, const int32_t* n_tile_active, void* workspace,
                                 size_t workspace_bytes, kvq_cuda_stream stream) {
  if (n_requests < 0) return fail(KVQ_ERR_BAD_ARG, "n_requests %d", n_requests);
  if (n_loops < 1 || n_loops > 4)
    return fail(KVQ_ERR_UNSUPPORTED, "n_loops %d (the batched append takes chains of 1..4 loops)", n_loops);
  if (n_heads < 1 || n_heads > 1024) return fail(KVQ_ERR_BAD_ARG, "n_heads %d", n_heads);
  if (head_dim != kD) return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d (kernels support 128)", head_dim);
  const size_t need = kvq_append_batch_workspace_bytes(n_requests);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return fail(KVQ_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", need);
  if (n_requests == 0) return ok();
  if (!reqs || !xk_tile || !xv_tile || !tile_active || !n_tile_active)
    return fail(KVQ_ERR_BAD_ARG, "NULL argument");
  if (!aligned16(reqs)) return fail(KVQ_ERR_MISALIGNED, "reqs must be 16-byte aligned");
  int sms = 0;
  kvq_status st = current_sms(&sms);
  if (st != KVQ_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int32_t* err = reinterpret_cast<int32_t*>(ws);
  int32_t* prefix = reinterpret_cast<int32_t*>(ws + 16);
  int32_t* skip = reinterpret_cast<int32_t*>(ws + 16 + round16(size_t(n_requests + 1) * 4));
  cudaError_t e = cudaMemsetAsync(err, 0, 16, s);
  if (e != cudaSuccess) return cuda_status(e, "clear error word");
  AppendBatchArgs pa;
  memset(&pa, 0, sizeof pa);
  pa.reqs = reqs;
  pa.n_requests = n_requests;
  pa.n_loops = n_loops;
  pa.H = n_heads;
  pa.tile_active = tile_active;
  pa.n_tile_active = n_tile_active;
  pa.skip = skip;
  pa.err = err;
  e = launch_append_batch_prep(pa, s);
  if (e != cudaSuccess) return cuda_status(e, "append preparation launch");
  // the table now counts the tile: encode the last tile of every loop, K and V
  for (int r = 0; r < n_loops; ++r) {
    for (int kind = KVQ_K; kind <= KVQ_V; ++kind) {
      CodecArgs a;
      memset(&a, 0, sizeof a);
      a.reqs = reqs;
      a.x = (kind == KVQ_K ? xk_tile : xv_tile) + size_t(r) * n_requests;
      a.n_requests = n_requests;
      a.H = n_heads;
      a.kind = kind;
      a.loop = r;
      a.append = 1;
      a.skip = skip;
      a.err = err;
      e = launch_codec(a, kind == KVQ_K ? kModeEncK : kModeEncV, prefix, sms, s);
      if (e != cudaSuccess) return cuda_status(e, "append encode launch");
    }
  }
  return ok();
}

kvq_status kvq_reconstruct(const kvq_stream* loops, int depth, uint16_t* out, kvq_cuda_stream stream) {
  Chain C;
  kvq_status st = build_chain(loops, depth, &C, "loops");
  if (st != KVQ_OK) return st;
  if (C.n_tokens == 0) return ok();
  if (out == nullptr) return fail(KVQ_ERR_BAD_ARG, "out is NULL");
  if (!aligned16(out)) return fail(KVQ_ERR_MISALIGNED, "out must be 16-byte aligned");
  CodecArgs a;
  memset(&a, 0, sizeof a);
  a.H = loops[0].n_heads;
  a.kind = loops[0].kind;
  a.loop = depth;
  a.one.n_tokens = loops[0].n_tokens;
  a.one.n_loops = depth;
  for (int j = 0; j < depth; ++j) to_loop_ref(&loops[j], &a.one.loop[j]);
  a.one_out = out;
  a.nvfp4 = nvfp4_mask(loops, depth);
  return run_single(a, kModeRecon, reinterpret_cast<cudaStream_t>(stream), "reconstruct launch");
}

size_t kvq_batch_workspace_bytes(int n_requests) {
  if (n_requests < 0) return 0;
  return 16 + round16(size_t(n_requests + 1) * 4);
}

static kvq_status check_batch(const kvq_request* reqs, int n_requests, int n_heads, int head_dim, int kind,
                              const void* ptrs, void* workspace, size_t workspace_bytes) {
  if (n_requests < 0) return fail(KVQ_ERR_BAD_ARG, "n_requests %d", n_requests);
  if (n_heads < 1 || n_heads > 1024) return fail(KVQ_ERR_BAD_ARG, "n_heads %d", n_heads);
  if (head_dim != kD) return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d (kernels support 128)", head_dim);
  if (kind != KVQ_K && kind != KVQ_V) return fail(KVQ_ERR_BAD_ARG, "kind %d", kind);
  if (n_requests == 0) return KVQ_OK;
  if (reqs == nullptr || ptrs == nullptr) return fail(KVQ_ERR_BAD_ARG, "NULL reqs or pointer array");
  if (!aligned16(reqs)) return fail(KVQ_ERR_MISALIGNED, "reqs must be 16-byte aligned");
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < kvq_batch_workspace_bytes(n_requests))
    return fail(KVQ_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", kvq_batch_workspace_bytes(n_requests));
  return KVQ_OK;
}

kvq_status kvq_encode_batch(const kvq_request* reqs, int n_requests, int n_heads, int head_dim, int kind, int loop,
                            const uint16_t* const* x, void* workspace, size_t workspace_bytes,
                            kvq_cuda_stream stream) {
  return kvq_encode_batch_ex(reqs, n_requests, n_heads, head_dim, kind, loop, x, 0u, workspace, workspace_bytes,
                             stream);
}

kvq_status kvq_encode_batch_ex(const kvq_request* reqs, int n_requests, int n_heads, int head_dim, int kind,
                               int loop, const uint16_t* const* x, uint32_t nvfp4_loops, void* workspace,
                               size_t workspace_bytes, kvq_cuda_stream stream) {
  kvq_status st = check_batch(reqs, n_requests, n_heads, head_dim, kind, x, workspace, workspace_bytes);
  if (st != KVQ_OK) return st;
  if (loop < 0 || loop >= KVQ_MAX_LOOPS) return fail(KVQ_ERR_BAD_ARG, "loop %d", loop);
  if ((nvfp4_loops & 1u) || (nvfp4_loops >> KVQ_MAX_LOOPS))
    return fail(KVQ_ERR_BAD_ARG, "nvfp4_loops 0x%x: the base is INT4 and at most %d loops", nvfp4_loops,
                KVQ_MAX_LOOPS);
  if (n_requests == 0) return ok();
  int sms = 0;
  st = current_sms(&sms);
  if (st != KVQ_OK) return st;
  CodecArgs a;
  memset(&a, 0, sizeof a);
  a.reqs = reqs;
  a.x = x;
  a.n_requests = n_requests;
  a.H = n_heads;
  a.kind = kind;
  a.loop = loop;
  a.nvfp4 = nvfp4_loops & ((2u << loop) - 1u);  // loops 0 .. loop
  char* ws = static_cast<char*>(workspace);
  a.err = reinterpret_cast<int32_t*>(ws);
  int32_t* prefix = reinterpret_cast<int32_t*>(ws + 16);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(a.err, 0, 16, s);
  if (e != cudaSuccess) return cuda_status(e, "clear error word");
  if (loop > 0) {
    e = launch_codec(a, kModeTileDir, prefix, sms, s);
    if (e != cudaSuccess) return cuda_status(e, "tile_dir launch");
  }
  return cuda_status(launch_codec(a, kind == KVQ_K ? kModeEncK : kModeEncV, prefix, sms, s), "encode launch");
}

kvq_status kvq_reconstruct_batch(const kvq_request* reqs, int n_requests, int n_heads, int head_dim, int kind,
                                 int depth, uint16_t* const* out, void* workspace, size_t workspace_bytes,
                                 kvq_cuda_stream stream) {
  return kvq_reconstruct_batch_ex(reqs, n_requests, n_heads, head_dim, kind, depth, out, 0u, workspace,
                                  workspace_bytes, stream);
}

kvq_status kvq_reconstruct_batch_ex(const kvq_request* reqs, int n_requests, int n_heads, int head_dim, int kind,
                                    int depth, uint16_t* const* out, uint32_t nvfp4_loops, void* workspace,
                                    size_t workspace_bytes, kvq_cuda_stream stream) {
  kvq_status st = check_batch(reqs, n_requests, n_heads, head_dim, kind, out, workspace, workspace_bytes);
  if (st != KVQ_OK) return st;
  if (depth < 1 || depth > KVQ_MAX_LOOPS) return fail(KVQ_ERR_BAD_ARG, "depth %d", depth);
  if ((nvfp4_loops & 1u) || (nvfp4_loops >> KVQ_MAX_LOOPS))
    return fail(KVQ_ERR_BAD_ARG, "nvfp4_loops 0x%x: the base is INT4 and at most %d loops", nvfp4_loops,
                KVQ_MAX_LOOPS);
  if (n_requests == 0) return ok();
  int sms = 0;
  st = current_sms(&sms);
  if (st != KVQ_OK) return st;
  CodecArgs a;
  memset(&a, 0, sizeof a);
  a.reqs = reqs;
  a.out = out;
  a.n_requests = n_requests;
  a.H = n_heads;
  a.kind = kind;
  a.loop = depth;
  a.nvfp4 = nvfp4_loops & ((1u << depth) - 1u);  // loops 0 .. depth-1
  char* ws = static_cast<char*>(workspace);
  a.err = reinterpret_cast<int32_t*>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(a.err, 0, 16, s);
  if (e != cudaSuccess) return cuda_status(e, "clear error word");
  return cuda_status(launch_codec(a, kModeRecon, reinterpret_cast<int32_t*>(ws + 16), sms, s), "reconstruct launch");
}

kvq_status kvq_request_fill(const kvq_stream* k_loops, const kvq_stream* v_loops, int n_loops, kvq_request* out) {
  if (out == nullptr || k_loops == nullptr || v_loops == nullptr) return fail(KVQ_ERR_BAD_ARG, "NULL argument");
  if (n_loops < 1 || n_loops > KVQ_MAX_LOOPS) return fail(KVQ_ERR_BAD_ARG, "n_loops %d", n_loops);
  memset(out, 0, sizeof *out);
  for (int j = 0; j < n_loops; ++j) {
    const kvq_stream* k = &k_loops[j];
    const kvq_stream* v = &v_loops[j];
    kvq_status st = check_planes(k, "k_loops[j]", true);
    if (st != KVQ_OK) return st;
    st = check_planes(v, "v_loops[j]", true);
    if (st != KVQ_OK) return st;
    if (k->kind != KVQ_K || v->kind != KVQ_V) return fail(KVQ_ERR_BAD_ARG, "loop %d: kinds must be K and V", j);
    if (k->n_rows != v->n_rows || k->n_tokens != v->n_tokens || k->n_heads != v->n_heads ||
        (k->active_idx == nullptr) != (v->active_idx == nullptr))
      return fail(KVQ_ERR_BAD_ARG, "loop %d: K and V streams disagree", j);
    if (k->n_tokens != k_loops[0].n_tokens) return fail(KVQ_ERR_BAD_ARG, "loop %d: n_tokens differs", j);
    if (j == 0 && k->active_idx != nullptr) return fail(KVQ_ERR_BAD_ARG, "loop 1 must be dense");
    kvq_loop_ref& L = out->loop[j];
    L.n_rows = k->n_rows;
    L.flags = loop_flags(k) | loop_flags(v);
    if (row_capacity(k) != row_capacity(v)) return fail(KVQ_ERR_BAD_ARG, "loop %d: K and V row capacities differ", j);
    L.row_cap = k->row_cap;
    L.kgroup_cap = k->row_cap > 0 ? k_groups_of(k_tile(k), k->row_cap, k->token_cap) : 0;
    L.active_idx = k->active_idx;
    L.tile_dir = k->tile_dir ? k->tile_dir : v->tile_dir;
    L.k_codes = k->codes;
    L.k_mins = k->mins;
    L.k_scales = k->scales;
    L.v_codes = v->codes;
    L.v_mins = v->mins;
    L.v_scales = v->scales;
  }
  out->n_tokens = k_loops[0].n_tokens;
  out->n_loops = n_loops;
  return ok();
}

size_t kvq_decode_attn_workspace_bytes(int n_requests, int n_heads, int n_q_heads, int head_dim) {
  (void)head_dim;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int sms = sm_count(dev);
  if (n_requests < 0 || n_heads < 1 || n_q_heads < 1 || sms <= 0) return 0;
  return ws_bytes(n_requests, n_heads, n_q_heads, sms * kMaxCtasPerSm);
}

// Arguments of one packed attention call with its workspace at `ws` (sized by
// ws_bytes for sms * kMaxCtasPerSm CTAs); algo is SIMT or MMA.
static void attention_args(AttnArgs& a, const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads, int depth,
                           const uint16_t* q, float softmax_scale, float* out, char* ws, int algo, bool nvfp4_hint,
                           int dev, int sms) {
  memset(&a, 0, sizeof a);
  a.reqs = reqs;
  a.n_requests = n_requests;
  a.H = n_heads;
  a.Hq = n_q_heads;
  a.g = n_q_heads / n_heads;
  a.depth = depth;
  a.nvfp4 = nvfp4_hint ? 1 : 0;
  a.refuse_nvfp4 = (algo == KVQ_ATTN_MMA && !nvfp4_hint) ? 1 : 0;
  a.n_ctas = attn_ctas(algo, dev);
  a.q = q;
  a.scale = softmax_scale;
  a.out = out;
  a.err = reinterpret_cast<int32_t*>(ws);
  a.flags = reinterpret_cast<int32_t*>(ws + 4);  // cleared with the error word
  a.prefix = reinterpret_cast<int32_t*>(ws + ws_prefix_offset());
  a.partials = reinterpret_cast<float*>(ws + ws_partials_offset(n_requests));
  a.stats = reinterpret_cast<float2*>(ws + ws_stats_offset(n_requests, n_heads, sms * kMaxCtasPerSm));
}

// Plan, attention, split-unit merge and (when asked) the BF16 segments, on a
// cleared error word.
static kvq_status attention_launches(const AttnArgs& a0, int algo, bool segments, cudaStream_t s) {
  AttnArgs a = a0;
  // the tcgen05 kernel runs one CTA of the work split per block, one block per SM
  // (attn_ctas counts two per SM for the tensor-core kernels)
  if (runs_tcgen05(a, algo == KVQ_ATTN_MMA)) a.n_ctas = a0.n_ctas / 2;
  cudaError_t e = launch_plan(a, s);
  if (e != cudaSuccess) return cuda_status(e, "plan launch");
  if (algo == KVQ_ATTN_MMA && a.nvfp4 && !a.general && !a.tcgen05) {
    // the table may hold NVFP4 loops: the INT4 kernel, then the NVFP4-reading
    // one; the plan's flag makes exactly one of them work, the other leaves
    AttnArgs t = a;
    t.nvfp4 = 0;
    t.dispatch = 1;
    e = launch_attn_mma(t, s);
    if (e != cudaSuccess) return cuda_status(e, "attention launch");
    a.dispatch = 2;
  }
  e = (algo == KVQ_ATTN_SIMT) ? launch_attn_simt(a, s) : launch_attn_mma(a, s);
  if (e != cudaSuccess) return cuda_status(e, "attention launch");
  e = launch_combine(a, s);
  if (e != cudaSuccess) return cuda_status(e, "combine launch");
  if (segments) {
    e = launch_segments(a, s);
    if (e != cudaSuccess) return cuda_status(e, "segment launch");
  }
  return ok();
}

kvq_status kvq_decode_attn_packed_ex(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads,
                                     int head_dim, int depth, const uint16_t* q, float softmax_scale, float* out,
                                     void* workspace, size_t workspace_bytes, int algo, kvq_cuda_stream stream) {
  if (n_requests < 0) return fail(KVQ_ERR_BAD_ARG, "n_requests %d", n_requests);
  if (n_heads < 1 || n_heads > 1024) return fail(KVQ_ERR_BAD_ARG, "n_heads %d", n_heads);
  if (n_q_heads < n_heads || n_q_heads % n_heads != 0)
    return fail(KVQ_ERR_BAD_ARG, "n_q_heads %d is not a multiple of n_heads %d", n_q_heads, n_heads);
  const int g = n_q_heads / n_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return fail(KVQ_ERR_UNSUPPORTED, "query heads per KV head %d (supported: 1, 2, 4, 8)", g);
  if (head_dim != kD) return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d (kernels support 128)", head_dim);
  if (depth < 1 || depth > KVQ_MAX_LOOPS) return fail(KVQ_ERR_BAD_ARG, "depth %d", depth);
  if (!(softmax_scale > 0.0f) || softmax_scale > 1e30f) return fail(KVQ_ERR_BAD_ARG, "softmax_scale");
  const bool nvfp4_hint = (algo & KVQ_ATTN_NVFP4) != 0;
  algo &= ~KVQ_ATTN_NVFP4;
  if (algo < KVQ_ATTN_AUTO || algo > KVQ_ATTN_TCGEN05) return fail(KVQ_ERR_BAD_ARG, "algo %d", algo);
  const bool general = algo == KVQ_ATTN_MMA_GENERAL;
  const bool tcgen05 = algo == KVQ_ATTN_TCGEN05;
  if (general || tcgen05) algo = KVQ_ATTN_MMA;
  if (n_requests == 0) return ok();
  if (!reqs || !q || !out) return fail(KVQ_ERR_BAD_ARG, "NULL reqs, q or out");
  if (!aligned16(reqs) || !aligned16(q) || !aligned16(out))
    return fail(KVQ_ERR_MISALIGNED, "reqs, q and out must be 16-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
  const int sms = sm_count(dev);
  if (sms <= 0) return fail(KVQ_ERR_CUDA, "cannot read the SM count of device %d", dev);
  const size_t need = ws_bytes(n_requests, n_heads, n_q_heads, sms * kMaxCtasPerSm);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return fail(KVQ_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", need);
  if (algo == KVQ_ATTN_AUTO) algo = depth <= kMmaMaxDepth ? KVQ_ATTN_MMA : KVQ_ATTN_SIMT;
  if (algo == KVQ_ATTN_MMA && depth > kMmaMaxDepth)
    return fail(KVQ_ERR_UNSUPPORTED, "the tensor-core kernel reads depth <= %d (got %d)", kMmaMaxDepth, depth);

  AttnArgs a;
  attention_args(a, reqs, n_requests, n_heads, n_q_heads, depth, q, softmax_scale, out, static_cast<char*>(workspace),
                 algo, nvfp4_hint, dev, sms);
  a.general = general ? 1 : 0;
  a.tcgen05 = tcgen05 ? 1 : 0;
  a.clear_err = 1;  // the plan kernel clears the error word and flags first
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return attention_launches(a, algo, true, s);
}

kvq_status kvq_decode_attn_packed(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads,
                                  int head_dim, int depth, const uint16_t* q, float softmax_scale, float* out,
                                  void* workspace, size_t workspace_bytes, kvq_cuda_stream stream) {
  return kvq_decode_attn_packed_ex(reqs, n_requests, n_heads, n_q_heads, head_dim, depth, q, softmax_scale, out,
                                   workspace, workspace_bytes, KVQ_ATTN_AUTO, stream);
}

// ---------------------------------------------------------------- sparse decode attention

static size_t sparse_attn_part(int n_requests, int n_heads, int n_q_heads) {
  return (kvq_decode_attn_workspace_bytes(n_requests, n_heads, n_q_heads, kD) + 255) / 256 * 256;
}

size_t kvq_sparse_workspace_bytes(int n_requests, int n_heads, int n_q_heads, int head_dim, int max_tokens) {
  (void)head_dim;
  if (n_requests < 0 || n_heads < 1 || n_q_heads < 1 || max_tokens < 0) return 0;
  return sparse_attn_part(n_requests, n_heads, n_q_heads) + size_t(n_requests) * n_q_heads * size_t(max_tokens) * 4;
}

static kvq_status check_sparse(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads, int head_dim,
                               int depth, const uint16_t* q, float softmax_scale, int n_select, int max_tokens) {
  if (n_requests < 0) return fail(KVQ_ERR_BAD_ARG, "n_requests %d", n_requests);
  if (n_heads < 1 || n_heads > 1024) return fail(KVQ_ERR_BAD_ARG, "n_heads %d", n_heads);
  if (n_q_heads < n_heads || n_q_heads % n_heads != 0)
    return fail(KVQ_ERR_BAD_ARG, "n_q_heads %d is not a multiple of n_heads %d", n_q_heads, n_heads);
  if (n_q_heads / n_heads > kMaxG) return fail(KVQ_ERR_UNSUPPORTED, "more than %d query heads per KV head", kMaxG);
  if (head_dim != kD) return fail(KVQ_ERR_UNSUPPORTED, "head_dim %d (kernels support 128)", head_dim);
  if (depth < 1 || depth > KVQ_MAX_LOOPS) return fail(KVQ_ERR_BAD_ARG, "depth %d", depth);
  if (!(softmax_scale > 0.0f) || softmax_scale > 1e30f) return fail(KVQ_ERR_BAD_ARG, "softmax_scale");
  if (n_select < 0) return fail(KVQ_ERR_BAD_ARG, "n_select %d", n_select);
  if (max_tokens < 0 || max_tokens > (1 << 24)) return fail(KVQ_ERR_BAD_ARG, "max_tokens %d", max_tokens);
  if (n_requests > 0 && (!reqs || !q)) return fail(KVQ_ERR_BAD_ARG, "NULL reqs or q");
  if (n_requests > 0 && (!aligned16(reqs) || !aligned16(q))) return fail(KVQ_ERR_MISALIGNED, "reqs and q must be 16-byte aligned");
  return KVQ_OK;
}

kvq_status kvq_sparse_ref_state(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads, int head_dim,
                                int ref_depth, const uint16_t* q_ref, float softmax_scale, int n_select,
                                int max_tokens, int32_t* sel_idx, float* mass, float* o_ref, float* c_ref,
                                void* workspace, size_t workspace_bytes, kvq_cuda_stream stream) {
  kvq_status st = check_sparse(reqs, n_requests, n_heads, n_q_heads, head_dim, ref_depth, q_ref, softmax_scale,
                               n_select, max_tokens);
  if (st != KVQ_OK) return st;
  if (n_requests == 0) return ok();
  if ((n_select > 0 && !sel_idx) || !mass || !o_ref || !c_ref) return fail(KVQ_ERR_BAD_ARG, "NULL output");
  if (!aligned16(o_ref) || !aligned16(c_ref)) return fail(KVQ_ERR_MISALIGNED, "o_ref and c_ref must be 16-byte aligned");
  const size_t need = kvq_sparse_workspace_bytes(n_requests, n_heads, n_q_heads, head_dim, max_tokens);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need)
    return fail(KVQ_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", need);
  const size_t apart = sparse_attn_part(n_requests, n_heads, n_q_heads);
  float* logits = reinterpret_cast<float*>(static_cast<char*>(workspace) + apart);
  const int g = n_q_heads / n_heads;
  // the tensor-core attention writes every logit as it goes; the CUDA-core one
  // (depth > 4) does not, and a separate kernel recomputes them
  const bool tc = ref_depth <= kMmaMaxDepth && (g == 1 || g == 2 || g == 4 || g == 8) && aligned16(o_ref);
  if (tc) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
    const int sms = sm_count(dev);
    if (sms <= 0) return fail(KVQ_ERR_CUDA, "cannot read the SM count of device %d", dev);
    AttnArgs at;
    attention_args(at, reqs, n_requests, n_heads, n_q_heads, ref_depth, q_ref, softmax_scale, o_ref,
                   static_cast<char*>(workspace), KVQ_ATTN_MMA, true, dev, sms);
    at.logits = logits;
    at.logit_stride = max_tokens;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(at.err, 0, 16, s);
    if (e != cudaSuccess) return cuda_status(e, "clear error word");
    st = attention_launches(at, KVQ_ATTN_MMA, true, s);
  } else {  // the full attention at the reference depth: O_ref (and a cleared error word)
    st = kvq_decode_attn_packed_ex(reqs, n_requests, n_heads, n_q_heads, head_dim, ref_depth, q_ref, softmax_scale,
                                   o_ref, workspace, apart, KVQ_ATTN_AUTO | KVQ_ATTN_NVFP4, stream);
  }
  if (st != KVQ_OK) return st;
  SparseArgs a;
  memset(&a, 0, sizeof a);
  a.reqs = reqs;
  a.n_requests = n_requests;
  a.H = n_heads;
  a.Hq = n_q_heads;
  a.g = n_q_heads / n_heads;
  a.depth = ref_depth;
  a.max_tokens = max_tokens;
  a.n_select = n_select;
  a.q = q_ref;
  a.scale = softmax_scale;
  a.logits = logits;
  a.sel_idx = sel_idx;
  a.mass = mass;
  a.c_ref = c_ref;
  a.err = static_cast<int32_t*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(tc ? launch_sparse_select(a, s) : launch_sparse_select_path(a, s), "sparse reference launch");
}

static size_t sparse_mask_words(int max_tokens) { return 2 * ((size_t(max_tokens) + 63) / 64); }

size_t kvq_sparse_decode_workspace_bytes(int n_requests, int n_heads, int n_q_heads, int head_dim, int max_tokens) {
  (void)head_dim;
  if (n_requests < 0 || n_heads < 1 || n_q_heads < 1 || max_tokens < 0) return 0;
  return sparse_attn_part(n_requests, n_heads, n_q_heads) +
         size_t(n_requests) * n_q_heads * sparse_mask_words(max_tokens) * 4;
}

kvq_status kvq_sparse_decode_attn_ex(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads, int head_dim,
                                     int depth, const uint16_t* q, float softmax_scale, int n_select, int max_tokens,
                                     const int32_t* sel_idx, const float* mass, const float* o_ref, const float* c_ref,
                                     float* out, void* workspace, size_t workspace_bytes, int algo,
                                     kvq_cuda_stream stream) {
  kvq_status st = check_sparse(reqs, n_requests, n_heads, n_q_heads, head_dim, depth, q, softmax_scale, n_select,
                               max_tokens);
  if (st != KVQ_OK) return st;
  const bool nvfp4_hint = (algo & KVQ_ATTN_NVFP4) != 0;
  algo &= ~KVQ_ATTN_NVFP4;
  if (algo < KVQ_ATTN_AUTO || algo > KVQ_ATTN_MMA) return fail(KVQ_ERR_BAD_ARG, "algo %d", algo);
  if (n_requests == 0) return ok();
  if ((n_select > 0 && !sel_idx) || !mass || !o_ref || !c_ref || !out) return fail(KVQ_ERR_BAD_ARG, "NULL argument");
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < 16)
    return fail(KVQ_ERR_WORKSPACE, "workspace needs 16 bytes, 16-byte aligned");
  const int g = n_q_heads / n_heads;
  const bool tc_ok = depth <= kMmaMaxDepth && (g == 1 || g == 2 || g == 4 || g == 8) && aligned16(out);
  const size_t need = kvq_sparse_decode_workspace_bytes(n_requests, n_heads, n_q_heads, head_dim, max_tokens);
  if (algo == KVQ_ATTN_MMA && !tc_ok)
    return fail(KVQ_ERR_UNSUPPORTED,
                "the tensor-core path reads depth <= %d with 1, 2, 4 or 8 query heads per KV head and a 16-byte "
                "aligned out", kMmaMaxDepth);
  if (algo == KVQ_ATTN_MMA && workspace_bytes < need)
    return fail(KVQ_ERR_WORKSPACE, "the tensor-core path needs %zu bytes of workspace", need);
  // a small selection is cheaper gathered key by key than attended through key masks, which read every tile
  const bool small = (long long)n_select * 64 <= (long long)max_tokens;
  const bool tc = algo != KVQ_ATTN_SIMT && tc_ok && workspace_bytes >= need && !(algo == KVQ_ATTN_AUTO && small);
  SparseArgs a;
  memset(&a, 0, sizeof a);
  a.reqs = reqs;
  a.n_requests = n_requests;
  a.H = n_heads;
  a.Hq = n_q_heads;
  a.g = n_q_heads / n_heads;
  a.depth = depth;
  a.max_tokens = max_tokens;
  a.n_select = n_select;
  a.q = q;
  a.scale = softmax_scale;
  a.sel_idx = const_cast<int32_t*>(sel_idx);
  a.mass = const_cast<float*>(mass);
  a.c_ref = const_cast<float*>(c_ref);
  a.o_ref = o_ref;
  a.out = out;
  a.err = static_cast<int32_t*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(a.err, 0, 16, s);
  if (e != cudaSuccess) return cuda_status(e, "clear error word");
  if (!tc) return cuda_status(launch_sparse_attn(a, s), "sparse attention launch");

  // tensor-core path: key masks, the masked packed attention, the correction
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
  const int sms = sm_count(dev);
  if (sms <= 0) return fail(KVQ_ERR_CUDA, "cannot read the SM count of device %d", dev);
  char* ws = static_cast<char*>(workspace);
  const size_t apart = sparse_attn_part(n_requests, n_heads, n_q_heads);
  a.mask_words = int32_t(sparse_mask_words(max_tokens));
  a.sel_mask = reinterpret_cast<uint32_t*>(ws + apart);
  e = cudaMemsetAsync(a.sel_mask, 0, size_t(n_requests) * n_q_heads * a.mask_words * 4, s);
  if (e != cudaSuccess) return cuda_status(e, "clear key masks");
  e = launch_sparse_mask(a, s);
  if (e != cudaSuccess) return cuda_status(e, "key mask launch");
  AttnArgs at;
  attention_args(at, reqs, n_requests, n_heads, n_q_heads, depth, q, softmax_scale, out, ws, KVQ_ATTN_MMA, nvfp4_hint,
                 dev, sms);
  at.sel_mask = a.sel_mask;
  at.mask_words = a.mask_words;
  a.stats = at.stats;
  a.refuse_nvfp4 = at.refuse_nvfp4;
  st = attention_launches(at, KVQ_ATTN_MMA, false, s);
  if (st != KVQ_OK) return st;
  return cuda_status(launch_sparse_epilogue(a, s), "sparse epilogue launch");
}

kvq_status kvq_sparse_decode_attn(const kvq_request* reqs, int n_requests, int n_heads, int n_q_heads, int head_dim,
                                  int depth, const uint16_t* q, float softmax_scale, int n_select, int max_tokens,
                                  const int32_t* sel_idx, const float* mass, const float* o_ref, const float* c_ref,
                                  float* out, void* workspace, size_t workspace_bytes, kvq_cuda_stream stream) {
  return kvq_sparse_decode_attn_ex(reqs, n_requests, n_heads, n_q_heads, head_dim, depth, q, softmax_scale, n_select,
                                   max_tokens, sel_idx, mass, o_ref, c_ref, out, workspace, workspace_bytes,
                                   KVQ_ATTN_AUTO | KVQ_ATTN_NVFP4, stream);
}

}  // extern "C"
