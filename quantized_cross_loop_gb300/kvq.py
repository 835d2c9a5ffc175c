"""Thin ctypes binding over libkvq.so (include/kvq.h).

Argument marshalling only: PyTorch supplies device memory and the current
CUDA stream; every step of the path runs in the library's kernels. The
library is loaded on first use; if it is missing the call raises KvqError.
There is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvq.so")

KVQ_K = 0
KVQ_V = 1
KVQ_GROUP = 64
KVQ_TILE = 64
KVQ_MAX_LOOPS = 8
KVQ_FORMAT_VERSION = 1
PLANE_CODES, PLANE_MINS, PLANE_SCALES, PLANE_INDEX, PLANE_TILE_DIR = range(5)
ATTN_AUTO, ATTN_SIMT, ATTN_MMA, ATTN_MMA_GENERAL, ATTN_TCGEN05 = 0, 1, 2, 3, 4
ATTN_NVFP4 = 8  # OR-ed into algo: the table may hold NVFP4 residual loops
KVQ_KGROUP_COMPACT, KVQ_KGROUP_TILE = 0, 1  # K groups: 64 stored rows / the stored rows of one 64-token tile
KVQ_LOOP_K_TILE, KVQ_LOOP_K_NVFP4, KVQ_LOOP_V_NVFP4 = 1, 2, 4
KVQ_FMT_INT4, KVQ_FMT_NVFP4 = 0, 1  # residual formats: affine INT4 / E2M1 + E4M3 per 16 + FP32 per stream

EXPORTED = (
    "kvq_stream_init", "kvq_plane_bytes", "kvq_stream_payload_bytes", "kvq_encode_base", "kvq_encode_residual",
    "kvq_build_tile_dir", "kvq_reconstruct", "kvq_request_fill", "kvq_decode_attn_workspace_bytes",
    "kvq_decode_attn_packed", "kvq_decode_attn_packed_ex", "kvq_status_string", "kvq_last_error", "kvq_version",
    "kvq_batch_workspace_bytes", "kvq_encode_batch", "kvq_reconstruct_batch", "kvq_launch_count",
    "kvq_decode_attn_packed_noalloc", "kvq_sparse_workspace_bytes", "kvq_sparse_ref_state",
    "kvq_sparse_decode_attn", "kvq_stream_payload_bytes_ex", "kvq_stream_set_format", "kvq_encode_batch_ex",
    "kvq_reconstruct_batch_ex", "kvq_stream_set_capacity", "kvq_append_workspace_bytes", "kvq_append_tile",
    "kvq_append_batch_workspace_bytes", "kvq_append_tile_batch", "kvq_sparse_decode_workspace_bytes",
    "kvq_sparse_decode_attn_ex",
)


class KvqError(RuntimeError):
    pass


class kvq_stream(ctypes.Structure):
    _fields_ = [
        ("version", ctypes.c_uint32),
        ("bits", ctypes.c_uint8),
        ("kind", ctypes.c_uint8),
        ("group", ctypes.c_uint16),
        ("nibble_order", ctypes.c_uint8),
        ("kgroup", ctypes.c_uint8),
        ("format", ctypes.c_uint8),
        ("reserved", ctypes.c_uint8),
        ("n_rows", ctypes.c_int32),
        ("n_tokens", ctypes.c_int32),
        ("n_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("codes", ctypes.c_void_p),
        ("mins", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("active_idx", ctypes.c_void_p),
        ("tile_dir", ctypes.c_void_p),
        ("row_cap", ctypes.c_int32),
        ("token_cap", ctypes.c_int32),
    ]


class kvq_loop_ref(ctypes.Structure):
    _fields_ = [
        ("n_rows", ctypes.c_int32),
        ("flags", ctypes.c_int32),
        ("active_idx", ctypes.c_void_p),
        ("tile_dir", ctypes.c_void_p),
        ("k_codes", ctypes.c_void_p),
        ("k_mins", ctypes.c_void_p),
        ("k_scales", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("v_mins", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
        ("row_cap", ctypes.c_int32),
        ("kgroup_cap", ctypes.c_int32),
    ]


class kvq_request(ctypes.Structure):
    _fields_ = [
        ("n_tokens", ctypes.c_int32),
        ("n_loops", ctypes.c_int32),
        ("loop", kvq_loop_ref * KVQ_MAX_LOOPS),
        ("n_sink", ctypes.c_int32),
        ("n_tail", ctypes.c_int32),
        ("sink_k", ctypes.c_void_p),
        ("sink_v", ctypes.c_void_p),
        ("tail_k", ctypes.c_void_p),
        ("tail_v", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def lib():
    """Load libkvq.so (raises KvqError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise KvqError(f"{LIB_PATH} is missing: build it with quantized_cross_loop_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            P = ctypes.POINTER
            L.kvq_stream_init.argtypes = [P(kvq_stream), i32, i32, i32, i32, i32]
            L.kvq_plane_bytes.argtypes = [P(kvq_stream), i32]
            L.kvq_plane_bytes.restype = sz
            L.kvq_stream_payload_bytes.argtypes = [i32, i32, i32, i32, i32]
            L.kvq_stream_payload_bytes.restype = ctypes.c_int64
            L.kvq_stream_payload_bytes_ex.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
            L.kvq_stream_set_format.argtypes = [P(kvq_stream), i32]
            L.kvq_stream_set_capacity.argtypes = [P(kvq_stream), i32, i32]
            L.kvq_append_workspace_bytes.argtypes = [i32]
            L.kvq_append_workspace_bytes.restype = sz
            L.kvq_append_tile.argtypes = [P(kvq_stream), i32, vp, vp, vp, vp, sz, vp]
            L.kvq_append_batch_workspace_bytes.argtypes = [i32]
            L.kvq_append_batch_workspace_bytes.restype = sz
            L.kvq_append_tile_batch.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
            L.kvq_stream_payload_bytes_ex.restype = ctypes.c_int64
            L.kvq_encode_base.argtypes = [vp, P(kvq_stream), vp]
            L.kvq_encode_residual.argtypes = [vp, P(kvq_stream), i32, P(kvq_stream), vp]
            L.kvq_build_tile_dir.argtypes = [vp, i32, i32, vp, vp]
            L.kvq_reconstruct.argtypes = [P(kvq_stream), i32, vp, vp]
            L.kvq_request_fill.argtypes = [P(kvq_stream), P(kvq_stream), i32, P(kvq_request)]
            L.kvq_decode_attn_workspace_bytes.argtypes = [i32, i32, i32, i32]
            L.kvq_decode_attn_workspace_bytes.restype = sz
            L.kvq_decode_attn_packed.argtypes = [vp, i32, i32, i32, i32, i32, vp, ctypes.c_float, vp, vp, sz, vp]
            L.kvq_decode_attn_packed_ex.argtypes = [vp, i32, i32, i32, i32, i32, vp, ctypes.c_float, vp, vp, sz,
                                                    i32, vp]
            L.kvq_sparse_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
            L.kvq_sparse_workspace_bytes.restype = sz
            L.kvq_sparse_ref_state.argtypes = [vp, i32, i32, i32, i32, i32, vp, ctypes.c_float, i32, i32, vp, vp, vp,
                                               vp, vp, sz, vp]
            L.kvq_sparse_decode_attn.argtypes = [vp, i32, i32, i32, i32, i32, vp, ctypes.c_float, i32, i32, vp, vp, vp,
                                                 vp, vp, vp, sz, vp]
            L.kvq_sparse_decode_attn_ex.argtypes = [vp, i32, i32, i32, i32, i32, vp, ctypes.c_float, i32, i32, vp, vp,
                                                    vp, vp, vp, vp, sz, i32, vp]
            L.kvq_sparse_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
            L.kvq_sparse_decode_workspace_bytes.restype = sz
            L.kvq_status_string.argtypes = [i32]
            L.kvq_status_string.restype = ctypes.c_char_p
            L.kvq_last_error.restype = ctypes.c_char_p
            L.kvq_version.restype = ctypes.c_uint32
            L.kvq_launch_count.restype = ctypes.c_uint64
            L.kvq_batch_workspace_bytes.argtypes = [i32]
            L.kvq_batch_workspace_bytes.restype = sz
            L.kvq_encode_batch.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, sz, vp]
            L.kvq_reconstruct_batch.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, sz, vp]
            L.kvq_encode_batch_ex.argtypes = [vp, i32, i32, i32, i32, i32, vp, ctypes.c_uint32, vp, sz, vp]
            L.kvq_reconstruct_batch_ex.argtypes = [vp, i32, i32, i32, i32, i32, vp, ctypes.c_uint32, vp, sz, vp]
            for name in ("kvq_stream_init", "kvq_encode_base", "kvq_encode_residual", "kvq_build_tile_dir",
                         "kvq_reconstruct", "kvq_request_fill", "kvq_decode_attn_packed",
                         "kvq_decode_attn_packed_ex", "kvq_encode_batch", "kvq_reconstruct_batch",
                         "kvq_stream_set_format", "kvq_encode_batch_ex", "kvq_reconstruct_batch_ex",
                         "kvq_stream_set_capacity", "kvq_append_tile", "kvq_append_tile_batch"):
                getattr(L, name).restype = ctypes.c_int32
            _lib = L
    return _lib


def _check(status: int, what: str):
    if status != 0:
        L = lib()
        raise KvqError(f"{what}: {L.kvq_status_string(status).decode()} ({L.kvq_last_error().decode()})")


def _stream_handle(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _require_cuda(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise KvqError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise KvqError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise KvqError(f"{name} must be {dtype}, got {t.dtype}")


class Stream:
    """One encoded loop of K or V: the planes (torch tensors on the device) and
    the C descriptor pointing at them."""

    def __init__(self, kind: int, n_rows: int, n_tokens: int, n_heads: int, head_dim: int, device,
                 active: torch.Tensor | None = None, alloc=None, shared_index=None, kgroup: int = KVQ_KGROUP_COMPACT,
                 fmt: int = KVQ_FMT_INT4, row_cap: int = 0, token_cap: int = 0):
        """row_cap, token_cap: room to grow (kvq_append_tile); 0 = exactly n_rows / n_tokens."""
        self.desc = kvq_stream()
        _check(lib().kvq_stream_init(ctypes.byref(self.desc), kind, n_rows, n_tokens, n_heads, head_dim),
               "kvq_stream_init")
        self.desc.kgroup = kgroup
        _check(lib().kvq_stream_set_format(ctypes.byref(self.desc), fmt), "kvq_stream_set_format")
        if row_cap or token_cap:
            _check(lib().kvq_stream_set_capacity(ctypes.byref(self.desc), row_cap, token_cap),
                   "kvq_stream_set_capacity")
        self.kind, self.n_rows, self.n_tokens, self.n_heads, self.head_dim = kind, n_rows, n_tokens, n_heads, head_dim
        self.kgroup, self.fmt = kgroup, fmt
        self.row_cap, self.token_cap = (row_cap or n_rows), (token_cap or n_tokens)

        def plane(p):
            nbytes = int(lib().kvq_plane_bytes(ctypes.byref(self.desc), p))
            if alloc is not None:
                return alloc(nbytes)
            return torch.empty(nbytes, dtype=torch.uint8, device=device)

        self.codes = plane(PLANE_CODES)
        self.mins = plane(PLANE_MINS)
        self.scales = plane(PLANE_SCALES)
        self.active = None
        self.tile_dir = None
        if shared_index is not None:  # K and V of one loop share the active set and its directory
            self.active, self.tile_dir = shared_index
        elif active is not None:
            buf = plane(PLANE_INDEX)
            buf.view(torch.int32)[:n_rows].copy_(active.to(device=device, dtype=torch.int32).reshape(-1))
            self.active = buf
            self.tile_dir = plane(PLANE_TILE_DIR)
        self.desc.codes = self.codes.data_ptr()
        self.desc.mins = self.mins.data_ptr()
        self.desc.scales = self.scales.data_ptr()
        self.desc.active_idx = None if self.active is None else self.active.data_ptr()
        self.desc.tile_dir = None if self.tile_dir is None else self.tile_dir.data_ptr()

    @property
    def sparse(self) -> bool:
        return self.active is not None

    # views with the logical plane shapes
    def codes_view(self):
        """uint8 [H, n_rows, D/2] (the live rows of the [H, row_cap, D/2] plane)."""
        full = self.codes[: self.n_heads * self.row_cap * self.head_dim // 2].view(self.n_heads, self.row_cap,
                                                                                   self.head_dim // 2)
        return full[:, : self.n_rows]

    def _groups(self, rows: int, tokens: int) -> int:
        if rows <= 0:
            return 0
        if self.kgroup == KVQ_KGROUP_TILE:
            return -(-tokens // KVQ_GROUP)
        return -(-rows // KVQ_GROUP)

    def param_shape(self, capacity: bool = False):
        rows = self.row_cap if capacity else self.n_rows
        if self.fmt == KVQ_FMT_NVFP4:  # E4M3 block scales (bytes)
            return (self.n_heads, rows, self.head_dim // 16)
        if self.kind == KVQ_K:
            return (self.n_heads, self._groups(rows, self.token_cap if capacity else self.n_tokens), self.head_dim)
        return (self.n_heads, rows, -(-self.head_dim // KVQ_GROUP))

    def _param_view(self, buf, dtype):
        full = self.param_shape(capacity=True)
        live = self.param_shape()
        return buf.view(dtype)[: math.prod(full)].view(full)[:, : live[1]]

    def mins_view(self):
        """INT4: FP16 mins (int16 bits); NVFP4: the E4M3 block scales (uint8 bits)."""
        return self._param_view(self.mins, torch.uint8 if self.fmt == KVQ_FMT_NVFP4 else torch.int16)

    def scales_view(self):
        """INT4: FP16 scales (int16 bits); NVFP4: the tensor scale (float32 [1])."""
        if self.fmt == KVQ_FMT_NVFP4:
            return self.scales.view(torch.float32)[:1]
        return self._param_view(self.scales, torch.int16)

    def active_view(self):
        return None if self.active is None else self.active.view(torch.int32)[: self.n_rows]

    def tile_dir_view(self):
        if self.tile_dir is None:
            return None
        return self.tile_dir.view(torch.int32)[: -(-self.n_tokens // KVQ_TILE) + 1]


def payload_bytes(kind: int, n_rows: int, n_heads: int, head_dim: int, sparse: bool, n_tokens: int | None = None,
                  kgroup: int = KVQ_KGROUP_COMPACT, fmt: int = KVQ_FMT_INT4) -> int:
    if n_tokens is None and kgroup == KVQ_KGROUP_COMPACT and fmt == KVQ_FMT_INT4:
        return int(lib().kvq_stream_payload_bytes(kind, n_rows, n_heads, head_dim, int(sparse)))
    T = n_rows if n_tokens is None else n_tokens
    return int(lib().kvq_stream_payload_bytes_ex(kind, n_rows, T, n_heads, head_dim, int(sparse), kgroup, fmt))


def kvq_encode_base(x: torch.Tensor, kind: int, stream=None, kgroup: int = KVQ_KGROUP_COMPACT,
                    token_cap: int = 0) -> Stream:
    """Encode the loop-1 base of K (kind=KVQ_K) or V from BF16 x [T, H, D]. The
    base is dense, so `kgroup` changes no byte; it is recorded with the stream.
    token_cap > T leaves room to append tiles (kvq_append_tile)."""
    _require_cuda(x, "x", torch.bfloat16)
    T, H, D = x.shape
    out = Stream(kind, T, T, H, D, x.device, kgroup=kgroup, row_cap=token_cap, token_cap=token_cap)
    _check(lib().kvq_encode_base(_dptr(x), ctypes.byref(out.desc), _stream_handle(stream)), "kvq_encode_base")
    return out


def kvq_encode_residual(x_r: torch.Tensor, prev: list, active: torch.Tensor | None = None, stream=None,
                        kgroup: int | None = None, fmt: int = KVQ_FMT_INT4, row_cap: int = 0,
                        token_cap: int = 0) -> Stream:
    """Encode loop len(prev)+1 of the chain `prev` from BF16 x_r [T, H, D];
    `active` (sorted int32 logical rows) makes it a compact sparse residual.
    `kgroup` (K only): KVQ_KGROUP_COMPACT or KVQ_KGROUP_TILE; default: the base's.
    `fmt`: KVQ_FMT_INT4 or KVQ_FMT_NVFP4 for this residual."""
    _require_cuda(x_r, "x_r", torch.bfloat16)
    T, H, D = x_r.shape
    kind = prev[0].kind
    n = T if active is None else int(active.numel())
    out = Stream(kind, n, T, H, D, x_r.device, active, kgroup=prev[0].kgroup if kgroup is None else kgroup, fmt=fmt,
                 row_cap=row_cap, token_cap=token_cap)
    arr = (kvq_stream * len(prev))(*[p.desc for p in prev])
    _check(lib().kvq_encode_residual(_dptr(x_r), arr, len(prev), ctypes.byref(out.desc), _stream_handle(stream)),
           "kvq_encode_residual")
    out._keep = list(prev)  # noqa: the chain must outlive the launch
    return out


def kvq_append_tile(streams: list, x_tile: list, tile_active: list, workspace: torch.Tensor | None = None,
                    stream=None):
    """Append one 64-token tile to the chain `streams` (one kind) in place: the
    flush of the BF16 tail into the packed form. x_tile[r]: BF16 [64, H, D] of
    loop r; tile_active[r]: int32 ascending positions 0..63 a sparse loop
    stores (None for a dense loop). Updates the streams' row and token counts."""
    n = len(streams)
    dev = streams[0].codes.device
    arr = (kvq_stream * n)(*[st.desc for st in streams])
    keep = []
    xs = (ctypes.c_void_p * n)()
    acts = (ctypes.c_void_p * n)()
    counts = (ctypes.c_int * n)()
    for r in range(n):
        _require_cuda(x_tile[r], f"x_tile[{r}]", torch.bfloat16)
        xs[r] = x_tile[r].data_ptr()
        a = tile_active[r]
        if a is None:
            acts[r] = None
            counts[r] = KVQ_TILE
        else:
            a = a.to(device=dev, dtype=torch.int32).contiguous()
            counts[r] = int(a.numel())
            if a.numel() == 0:  # an empty sparse tile still passes a valid pointer (NULL means dense)
                a = torch.zeros(1, dtype=torch.int32, device=dev)
            keep.append(a)
            acts[r] = a.data_ptr()
    if workspace is None:
        workspace = torch.empty(int(lib().kvq_append_workspace_bytes(n)), dtype=torch.uint8, device=dev)
    _check(lib().kvq_append_tile(arr, n, xs, acts, counts, _dptr(workspace), workspace.numel(), _stream_handle(stream)),
           "kvq_append_tile")
    for r, st in enumerate(streams):
        st.desc = arr[r]
        st.n_rows, st.n_tokens = arr[r].n_rows, arr[r].n_tokens
    streams[0]._append_keep = (keep, workspace)  # noqa: the launch reads them
    return workspace


def kvq_build_tile_dir(active: torch.Tensor, n_tokens: int, stream=None) -> torch.Tensor:
    _require_cuda(active, "active", torch.int32)
    out = torch.empty(-(-n_tokens // KVQ_TILE) + 1, dtype=torch.int32, device=active.device)
    _check(lib().kvq_build_tile_dir(_dptr(active), active.numel(), n_tokens, _dptr(out), _stream_handle(stream)),
           "kvq_build_tile_dir")
    return out


def kvq_reconstruct(streams: list, depth: int, stream=None) -> torch.Tensor:
    """BF16 [T, H, D] reconstruction of the chain at `depth`."""
    s0 = streams[0]
    out = torch.empty((s0.n_tokens, s0.n_heads, s0.head_dim), dtype=torch.bfloat16, device=s0.codes.device)
    arr = (kvq_stream * depth)(*[s.desc for s in streams[:depth]])
    _check(lib().kvq_reconstruct(arr, depth, _dptr(out), _stream_handle(stream)), "kvq_reconstruct")
    return out


class RequestTable:
    """Device array of kvq_request for a batch of requests (each a pair of K and
    V stream lists). Holds references to the streams so their planes outlive it."""

    def __init__(self, k_chains: list, v_chains: list, device=None, segments: list | None = None):
        """segments[b]: None, or (sink_k, sink_v, tail_k, tail_v) — BF16 device
        tensors [n, H, D] (or None) read by the attention next to the packed
        chain: the sink replaces the first tokens, the tail follows the last."""
        n = len(k_chains)
        host = (kvq_request * max(n, 1))()
        keep = []
        for b in range(n):
            ks, vs = k_chains[b], v_chains[b]
            ka = (kvq_stream * len(ks))(*[s.desc for s in ks])
            va = (kvq_stream * len(vs))(*[s.desc for s in vs])
            _check(lib().kvq_request_fill(ka, va, len(ks), ctypes.byref(host[b])), f"kvq_request_fill[{b}]")
            seg = segments[b] if segments is not None else None
            if seg is not None:
                sk, sv, tk, tv = seg
                for name, t in (("sink_k", sk), ("sink_v", sv), ("tail_k", tk), ("tail_v", tv)):
                    if t is not None:
                        _require_cuda(t, name, torch.bfloat16)
                        setattr(host[b], name, t.data_ptr() if t.numel() else None)
                        keep.append(t)
                host[b].n_sink = 0 if sk is None else int(sk.shape[0])
                host[b].n_tail = 0 if tk is None else int(tk.shape[0])
        raw = bytes(memoryview(host).cast("B"))
        if device is None:
            device = k_chains[0][0].codes.device if n else torch.device("cuda")
        self.table = torch.frombuffer(bytearray(raw), dtype=torch.uint8).to(device)
        self.n_requests = n
        self.has_nvfp4 = any(getattr(st, "fmt", KVQ_FMT_INT4) == KVQ_FMT_NVFP4
                             for chains in (k_chains, v_chains) for ch in chains for st in ch)
        self._keep = (k_chains, v_chains, keep)


def kvq_decode_attn_workspace_bytes(n_requests: int, n_heads: int, n_q_heads: int, head_dim: int) -> int:
    return int(lib().kvq_decode_attn_workspace_bytes(n_requests, n_heads, n_q_heads, head_dim))


def kvq_decode_attn_packed(table: RequestTable, q: torch.Tensor, depth: int, n_heads: int,
                           softmax_scale: float | None = None, algo: int = ATTN_AUTO, out: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """FP32 [B, Hq, D] decode attention of q [B, Hq, D] (BF16) over the packed
    chains of `table` at `depth`."""
    _require_cuda(q, "q", torch.bfloat16)
    B, Hq, D = q.shape
    if B != table.n_requests:
        raise KvqError(f"q has {B} requests, table has {table.n_requests}")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    need = kvq_decode_attn_workspace_bytes(B, n_heads, Hq, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if table.has_nvfp4:
        algo |= ATTN_NVFP4
    _check(lib().kvq_decode_attn_packed_ex(_dptr(table.table), B, n_heads, Hq, D, depth, _dptr(q),
                                           ctypes.c_float(softmax_scale), _dptr(out), _dptr(workspace),
                                           workspace.numel(), algo, _stream_handle(stream)),
           "kvq_decode_attn_packed")
    return out


def plane_bytes(kind: int, n_rows: int, n_tokens: int, n_heads: int, head_dim: int,
                kgroup: int = KVQ_KGROUP_COMPACT, fmt: int = KVQ_FMT_INT4, row_cap: int = 0, token_cap: int = 0) -> list:
    d = kvq_stream()
    _check(lib().kvq_stream_init(ctypes.byref(d), kind, n_rows, n_tokens, n_heads, head_dim), "kvq_stream_init")
    d.kgroup = kgroup
    _check(lib().kvq_stream_set_format(ctypes.byref(d), fmt), "kvq_stream_set_format")
    if row_cap or token_cap:
        _check(lib().kvq_stream_set_capacity(ctypes.byref(d), row_cap, token_cap), "kvq_stream_set_capacity")
    return [int(lib().kvq_plane_bytes(ctypes.byref(d), p)) for p in range(5)]


class PackedPool:
    """Device storage for the packed K/V chains of a batch of requests: one
    allocation, each request's planes contiguous and 256-byte aligned, located
    through the device request table (kvq_request per request).

    active_sets[b][r] is the sorted int32 active set of loop r of request b, or
    None for a dense loop (loop 0 must be dense). kgroup: the K grouping of
    every K stream (KVQ_KGROUP_COMPACT or KVQ_KGROUP_TILE). formats[r]: the
    format of loop r of K and V in every request (KVQ_FMT_INT4 default;
    KVQ_FMT_NVFP4 for residual loops r >= 1)."""

    ALIGN = 256

    def __init__(self, lengths: list, active_sets: list, n_heads: int, head_dim: int, n_loops: int, device,
                 kgroup: int = KVQ_KGROUP_COMPACT, formats: list | None = None, token_caps: list | None = None):
        """token_caps[b]: tokens request b may grow to by appended tiles (kvq_append_tile_batch);
        None: no room to grow."""
        device = torch.device(device)
        self.kgroup = kgroup
        self.token_caps = None if token_caps is None else [int(c) for c in token_caps]
        self.formats = [KVQ_FMT_INT4] * n_loops if formats is None else list(formats)
        if self.formats[0] != KVQ_FMT_INT4:
            raise KvqError("the base loop is INT4")
        self.nvfp4_mask = sum(1 << r for r, f in enumerate(self.formats) if f == KVQ_FMT_NVFP4)
        self.lengths = list(lengths)
        self.n_heads, self.head_dim, self.n_loops = n_heads, head_dim, n_loops
        # pass 1: sizes
        total = 0
        sizes = []
        for b, T in enumerate(self.lengths):
            per = []
            for r in range(n_loops):
                act = active_sets[b][r]
                n = T if act is None else int(act.numel())
                fm = self.formats[r]
                cap = 0 if self.token_caps is None else self.token_caps[b]
                k = plane_bytes(KVQ_K, n, T, n_heads, head_dim, kgroup, fm, cap, cap)
                v = plane_bytes(KVQ_V, n, T, n_heads, head_dim, KVQ_KGROUP_COMPACT, fm, cap, cap)
                per.append((n, k, v, act is not None))
                total += sum(self._up(x) for x in k[:3]) + sum(self._up(x) for x in v[:3])
                if act is not None:
                    total += self._up(k[PLANE_INDEX]) + self._up(k[PLANE_TILE_DIR])
            sizes.append(per)
        self.storage = torch.empty(max(total, self.ALIGN), dtype=torch.uint8, device=device)
        self.offset = 0
        self.payload_bytes = 0
        # pass 2: carve
        self.k_streams, self.v_streams = [], []
        for b, T in enumerate(self.lengths):
            ks, vs = [], []
            for r in range(n_loops):
                n, kb, vb, sparse = sizes[b][r]
                shared = None
                if sparse:
                    idx = self._take(kb[PLANE_INDEX])
                    idx.view(torch.int32)[:n].copy_(active_sets[b][r].to(device=device, dtype=torch.int32))
                    shared = (idx, self._take(kb[PLANE_TILE_DIR]))
                fm = self.formats[r]
                cap = 0 if self.token_caps is None else self.token_caps[b]
                ks.append(Stream(KVQ_K, n, T, n_heads, head_dim, device, alloc=self._take, shared_index=shared,
                                 kgroup=kgroup, fmt=fm, row_cap=cap, token_cap=cap))
                vs.append(Stream(KVQ_V, n, T, n_heads, head_dim, device, alloc=self._take, shared_index=shared,
                                 fmt=fm, row_cap=cap, token_cap=cap))
                self.payload_bytes += payload_bytes(KVQ_K, n, n_heads, head_dim, sparse, T, kgroup, fm)
                self.payload_bytes += payload_bytes(KVQ_V, n, n_heads, head_dim, False, T, KVQ_KGROUP_COMPACT, fm)
            self.k_streams.append(ks)
            self.v_streams.append(vs)
        self.table = RequestTable(self.k_streams, self.v_streams, device)
        self.workspace = torch.empty(int(lib().kvq_batch_workspace_bytes(len(self.lengths))), dtype=torch.uint8,
                                     device=device)

    def _up(self, n):
        return -(-n // self.ALIGN) * self.ALIGN

    def _take(self, nbytes):
        t = self.storage[self.offset:self.offset + nbytes]
        self.offset += self._up(nbytes)
        return t

    @property
    def n_requests(self):
        return len(self.lengths)

    def prepare_append(self, xk_tiles: list, xv_tiles: list, tile_active: list):
        """Device argument arrays of one append_tile call: xk_tiles[r][b], xv_tiles[r][b] are
        BF16 [64, H, D] device tensors of loop r and request b; tile_active[r][b] an int32
        tensor of positions 0..63 (sparse loop) or None (dense loop)."""
        dev = self.storage.device
        nb, nl = self.n_requests, self.n_loops
        keep, acts, counts = [], [], []
        for r in range(nl):
            for b in range(nb):
                a = tile_active[r][b]
                if a is None:
                    acts.append(0)
                    counts.append(KVQ_TILE)
                    continue
                a = a.to(device=dev, dtype=torch.int32).contiguous()
                counts.append(int(a.numel()))
                if a.numel() == 0:  # an empty sparse tile still passes a valid pointer (NULL means dense)
                    a = torch.zeros(1, dtype=torch.int32, device=dev)
                keep.append(a)
                acts.append(a.data_ptr())
        xk = pointer_array([xk_tiles[r][b] for r in range(nl) for b in range(nb)], dev)
        xv = pointer_array([xv_tiles[r][b] for r in range(nl) for b in range(nb)], dev)
        act = torch.tensor(acts, dtype=torch.int64, device=dev)
        cnt = torch.tensor(counts, dtype=torch.int32, device=dev)
        return (xk, xv, act, cnt, keep, xk_tiles, xv_tiles)

    def append_tile(self, xk_tiles: list = None, xv_tiles: list = None, tile_active: list = None,
                    workspace: torch.Tensor | None = None, stream=None, prepared=None) -> torch.Tensor:
        """Append one 64-token tile to every request (kvq_append_tile_batch), from the tiles
        (see prepare_append) or from a prepare_append result. The device table is updated
        in place; sync_counts() brings the new counts to the host objects. Returns the
        workspace (error word at offset 0)."""
        dev = self.storage.device
        args = prepared if prepared is not None else self.prepare_append(xk_tiles, xv_tiles, tile_active)
        xk, xv, act, cnt = args[:4]
        nb = self.n_requests
        if workspace is None:
            workspace = torch.empty(int(lib().kvq_append_batch_workspace_bytes(nb)), dtype=torch.uint8, device=dev)
        _check(lib().kvq_append_tile_batch(_dptr(self.table.table), nb, self.n_heads, self.head_dim, self.n_loops,
                                           _dptr(xk), _dptr(xv), _dptr(act), _dptr(cnt), _dptr(workspace),
                                           workspace.numel(), _stream_handle(stream)), "kvq_append_tile_batch")
        self._append_keep = args
        return workspace

    def sync_counts(self):
        """Read the device table back and update the host stream objects' row and token counts
        (a device-to-host read: for tests and tools, not for the serving path)."""
        raw = self.table.table.cpu().numpy().tobytes()
        host = (kvq_request * self.n_requests).from_buffer_copy(raw[: ctypes.sizeof(kvq_request) * self.n_requests])
        for b in range(self.n_requests):
            self.lengths[b] = host[b].n_tokens
            for r in range(self.n_loops):
                for st in (self.k_streams[b][r], self.v_streams[b][r]):
                    st.n_rows, st.n_tokens = host[b].loop[r].n_rows, host[b].n_tokens
                    st.desc.n_rows, st.desc.n_tokens = st.n_rows, st.n_tokens


def pointer_array(tensors: list, device) -> torch.Tensor:
    """Device int64 array of the tensors' data pointers (for the batched calls)."""
    return torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64, device=device)


def kvq_encode_batch(pool: PackedPool, kind: int, loop: int, x_ptrs: torch.Tensor, stream=None,
                     workspace: torch.Tensor | None = None):
    """Encode loop `loop` (0 = base) of `kind` for every request of the pool;
    x_ptrs: device int64 array of BF16 [T_b, H, D] source pointers. Calls that
    may run concurrently (on different streams) need their own `workspace`
    (kvq_batch_workspace_bytes(n_requests) bytes); the default is the pool's."""
    ws = pool.workspace if workspace is None else workspace
    _check(lib().kvq_encode_batch_ex(_dptr(pool.table.table), pool.n_requests, pool.n_heads, pool.head_dim, kind,
                                     loop, _dptr(x_ptrs), pool.nvfp4_mask, _dptr(ws), ws.numel(),
                                     _stream_handle(stream)), "kvq_encode_batch")


def kvq_reconstruct_batch(pool: PackedPool, kind: int, depth: int, out_ptrs: torch.Tensor, stream=None,
                          workspace: torch.Tensor | None = None):
    ws = pool.workspace if workspace is None else workspace
    _check(lib().kvq_reconstruct_batch_ex(_dptr(pool.table.table), pool.n_requests, pool.n_heads, pool.head_dim,
                                          kind, depth, _dptr(out_ptrs), pool.nvfp4_mask, _dptr(ws), ws.numel(),
                                          _stream_handle(stream)), "kvq_reconstruct_batch")


def launch_count() -> int:
    return int(lib().kvq_launch_count())


def kvq_decode_attn_packed_noalloc(table: RequestTable, q: torch.Tensor, depth: int, n_heads: int,
                                   softmax_scale: float | None = None, out: torch.Tensor | None = None,
                                   stream=None) -> torch.Tensor:
    """Same result as kvq_decode_attn_packed, for callers that cannot allocate:
    the library's static device scratch replaces the workspace. Calls that
    overlap on the GPU share that scratch and must be serialised."""
    _require_cuda(q, "q", torch.bfloat16)
    B, Hq, D = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    f = lib().kvq_decode_attn_packed_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int32
    _check(f(_dptr(table.table), B, n_heads, Hq, D, depth, _dptr(q), ctypes.c_float(softmax_scale), _dptr(out),
             _stream_handle(stream)), "kvq_decode_attn_packed_noalloc")
    return out


def attn_error_word(workspace: torch.Tensor) -> int:
    """The error word the attention kernels set in the workspace (reads the device)."""
    return int(workspace[:4].view(torch.int32).item())


# --------------------------------------------------------------------------- sparse decode attention


def kvq_sparse_workspace_bytes(n_requests: int, n_heads: int, n_q_heads: int, head_dim: int, max_tokens: int) -> int:
    return int(lib().kvq_sparse_workspace_bytes(n_requests, n_heads, n_q_heads, head_dim, max_tokens))


class SparseState:
    """Reference-loop state of sparse decode attention: selected positions
    [B, Hq, n_select] (-1 padded), mass [B, Hq], O_ref and C_ref [B, Hq, D]."""

    def __init__(self, sel_idx, mass, o_ref, c_ref, n_select, max_tokens, workspace):
        self.sel_idx, self.mass, self.o_ref, self.c_ref = sel_idx, mass, o_ref, c_ref
        self.n_select, self.max_tokens, self.workspace = n_select, max_tokens, workspace


def kvq_sparse_ref_state(table: RequestTable, q_ref: torch.Tensor, ref_depth: int, n_heads: int, n_select: int,
                         max_tokens: int, softmax_scale: float | None = None, workspace: torch.Tensor | None = None,
                         stream=None) -> SparseState:
    _require_cuda(q_ref, "q_ref", torch.bfloat16)
    B, Hq, D = q_ref.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    dev = q_ref.device
    sel = torch.empty((B, Hq, max(n_select, 1)), dtype=torch.int32, device=dev)
    mass = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    o_ref = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    c_ref = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    need = kvq_sparse_workspace_bytes(B, n_heads, Hq, D, max_tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check(lib().kvq_sparse_ref_state(_dptr(table.table), B, n_heads, Hq, D, ref_depth, _dptr(q_ref),
                                      ctypes.c_float(softmax_scale), n_select, max_tokens, _dptr(sel), _dptr(mass),
                                      _dptr(o_ref), _dptr(c_ref), _dptr(workspace), workspace.numel(),
                                      _stream_handle(stream)), "kvq_sparse_ref_state")
    return SparseState(sel[:, :, :n_select], mass, o_ref, c_ref, n_select, max_tokens, workspace)


def kvq_sparse_decode_workspace_bytes(n_requests: int, n_heads: int, n_q_heads: int, head_dim: int,
                                      max_tokens: int) -> int:
    return int(lib().kvq_sparse_decode_workspace_bytes(n_requests, n_heads, n_q_heads, head_dim, max_tokens))


def kvq_sparse_decode_attn(table: RequestTable, q: torch.Tensor, depth: int, n_heads: int, state: SparseState,
                           softmax_scale: float | None = None, out: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, algo: int = ATTN_AUTO, stream=None) -> torch.Tensor:
    """A later loop of sparse decode attention. With no workspace given, one of
    kvq_sparse_decode_workspace_bytes is allocated, so that AUTO takes the
    tensor-core path where it can; a 16-byte workspace selects the per-key
    kernel."""
    _require_cuda(q, "q", torch.bfloat16)
    B, Hq, D = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = kvq_sparse_decode_workspace_bytes(B, n_heads, Hq, D, state.max_tokens)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if table.has_nvfp4:
        algo |= ATTN_NVFP4
    sel = state.sel_idx.contiguous()
    _check(lib().kvq_sparse_decode_attn_ex(_dptr(table.table), B, n_heads, Hq, D, depth, _dptr(q),
                                           ctypes.c_float(softmax_scale), state.n_select, state.max_tokens,
                                           _dptr(sel), _dptr(state.mass), _dptr(state.o_ref), _dptr(state.c_ref),
                                           _dptr(out), _dptr(workspace), workspace.numel(), algo,
                                           _stream_handle(stream)),
           "kvq_sparse_decode_attn")
    return out
