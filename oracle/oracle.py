"""Python wrapper around the scalar CPU oracle (kvq_oracle.c).

TEST INFRASTRUCTURE ONLY. Only tests/, ``__graft_entry__.smoke()`` and the
cpu_baseline / reference leg of ``bench.py`` may import this module. It imports
nothing from the product package; the product package never imports it.

Arrays are numpy: BF16 and FP16 values travel as their uint16 bit patterns.
Layouts (head-major planes) are those written in kvq_oracle.c's header.

The chain helpers follow the FlashLoop RFC (vllm-rlt issue #156) §3.3: the
base is encoded from X1; loop r encodes X_r minus the reconstruction at depth
r-1, over all rows (dense) or over the sorted active rows (compact sparse).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB = os.path.join(_HERE, "liborc.so")
_lock = threading.Lock()
_lib = None

KIND_K = 0
KIND_V = 1
GROUP = 64
KGROUP_COMPACT = 0  # K groups: 64 consecutive stored rows (the codec PR's grouping)
KGROUP_TILE = 1     # K groups: the stored rows of one 64-token logical tile (page-local metadata)
FMT_INT4 = 0        # affine INT4 groups of 64, FP16 min and scale
FMT_NVFP4 = 1       # E2M1 elements, E4M3 scale per 16 channels, FP32 scale per stream (residuals only)


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c into liborc.so (plain scalar C, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = [
            "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-Wall", "-Wextra", "-Wno-unused-parameter", _SRC, "-o", tmp, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Stream(ctypes.Structure):
    _fields_ = [
        ("n", ctypes.c_int32),
        ("kgroup", ctypes.c_int32),
        ("active", ctypes.c_void_p),
        ("codes", ctypes.c_void_p),
        ("mins", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("fmt", ctypes.c_int32),
        ("_pad", ctypes.c_int32),
        ("bscale", ctypes.c_void_p),
        ("tscale", ctypes.c_void_p),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            L.orc_encode.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, i32, vp, vp, vp]
            L.orc_encode.restype = i32
            L.orc_encode_ex.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, i32, vp, vp, vp]
            L.orc_encode_ex.restype = i32
            L.orc_reconstruct.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(_Stream), vp]
            L.orc_reconstruct.restype = i32
            L.orc_attention.argtypes = [i32, i32, i32, i32, vp, vp, vp, ctypes.c_float, vp]
            L.orc_attention.restype = i32
            L.orc_attention_f32.argtypes = [i32, i32, i32, i32, vp, vp, vp, ctypes.c_float, vp]
            L.orc_attention_f32.restype = i32
            L.orc_decode_f32.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(_Stream), vp]
            L.orc_decode_f32.restype = i32
            L.orc_stream_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
            L.orc_stream_bytes.restype = i64
            L.orc_stream_bytes_ex.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
            L.orc_stream_bytes_ex.restype = i64
            L.orc_stream_bytes_nvfp4.argtypes = [i32, i32, i32, i32]
            L.orc_stream_bytes_nvfp4.restype = i64
            L.orc_encode_nvfp4.argtypes = [i32, i32, i32, i32, vp, vp, vp, i32, vp, vp, vp]
            L.orc_encode_nvfp4.restype = i32
            for name in ("orc_f32_to_e4m3_n", "orc_f32_to_e2m1_n"):
                getattr(L, name).argtypes = [vp, vp, i64]
                getattr(L, name).restype = None
            L.orc_e4m3_to_f32.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_to_f32.restype = ctypes.c_float
            L.orc_e2m1_to_f32.argtypes = [ctypes.c_uint8]
            L.orc_e2m1_to_f32.restype = ctypes.c_float
            for name in ("orc_f32_to_f16_n", "orc_f32_to_bf16_n", "orc_f16_to_f32_n"):
                getattr(L, name).argtypes = [vp, vp, i64]
                getattr(L, name).restype = None
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------- rounding helpers


def f32_to_f16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_f16_n(_ptr(x), _ptr(y), x.size)
    return y


def f32_to_bf16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_n(_ptr(x), _ptr(y), x.size)
    return y


def f16_bits_to_f32(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    y = np.empty(x.shape, dtype=np.float32)
    lib().orc_f16_to_f32_n(_ptr(x), _ptr(y), x.size)
    return y


def f32_to_e4m3_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint8)
    lib().orc_f32_to_e4m3_n(_ptr(x), _ptr(y), x.size)
    return y


def f32_to_e2m1_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint8)
    lib().orc_f32_to_e2m1_n(_ptr(x), _ptr(y), x.size)
    return y


def e4m3_bits_to_f32(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    table = np.array([lib().orc_e4m3_to_f32(i) for i in range(256)], dtype=np.float32)
    return table[b]


def e2m1_bits_to_f32(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    table = np.array([lib().orc_e2m1_to_f32(i) for i in range(16)], dtype=np.float32)
    return table[b & 15]


def bf16_bits_to_f32(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    return (x.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- codec


@dataclass
class Stream:
    """One encoded loop (base or residual) of K or V for one request/layer."""

    kind: int
    T: int
    H: int
    D: int
    n: int
    active: np.ndarray | None  # int32 [n] ascending, or None (dense)
    codes: np.ndarray  # uint8 [H, n, D/2]
    mins: np.ndarray  # uint16 (f16 bits): K [H, groups, D] (see param_shape); V [H, n, ceil(D/G)]
    scales: np.ndarray
    kgroup: int = KGROUP_COMPACT
    fmt: int = FMT_INT4
    bscale: np.ndarray | None = None  # NVFP4: uint8 E4M3 bits [H, n, D/16]
    tscale: np.ndarray | None = None  # NVFP4: float32 [1], the tensor scale

    def c_struct(self) -> _Stream:
        s = _Stream()
        s.n = self.n
        s.kgroup = self.kgroup
        s.fmt = self.fmt
        s.bscale = None if self.bscale is None else self.bscale.ctypes.data
        s.tscale = None if self.tscale is None else self.tscale.ctypes.data
        s.active = None if self.active is None else self.active.ctypes.data
        s.codes = self.codes.ctypes.data
        s.mins = self.mins.ctypes.data
        s.scales = self.scales.ctypes.data
        return s


def param_shape(kind: int, n: int, H: int, D: int, G: int = GROUP, T: int | None = None,
                kgroup: int = KGROUP_COMPACT, sparse: bool = False):
    """Param plane shape. K: one group per G stored rows, or, for a tile-grouped
    sparse stream, one per logical tile of G tokens (ceil(T/G)); V: per stored
    row and channel group."""
    if kind == KIND_K:
        if kgroup == KGROUP_TILE and sparse and n > 0:
            return (H, -(-T // G), D)
        return (H, -(-n // G), D)
    return (H, n, -(-D // G))


def encode(kind: int, x: np.ndarray, pred: np.ndarray | None = None, active: np.ndarray | None = None,
           G: int = GROUP, kgroup: int = KGROUP_COMPACT) -> Stream:
    """Encode one stream. x, pred: uint16 BF16 bits [T, H, D] (logical order).
    kgroup selects the K grouping of a sparse stream (V ignores it)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T, H, D = x.shape
    if pred is not None:
        pred = np.ascontiguousarray(pred, dtype=np.uint16)
        assert pred.shape == x.shape
    if active is not None:
        active = np.ascontiguousarray(active, dtype=np.int32)
        n = int(active.size)
    else:
        n = T
    codes = np.zeros((H, n, D // 2), dtype=np.uint8)
    mins = np.zeros(param_shape(kind, n, H, D, G, T, kgroup, active is not None), dtype=np.uint16)
    scales = np.zeros_like(mins)
    rc = lib().orc_encode_ex(kind, T, H, D, G, kgroup, _ptr(x), _ptr(pred), _ptr(active), n, _ptr(codes),
                             _ptr(mins), _ptr(scales))
    if rc != 0:
        raise ValueError(f"orc_encode failed with status {rc}")
    return Stream(kind, T, H, D, n, active, codes, mins, scales, kgroup)


def encode_nvfp4(kind: int, x: np.ndarray, pred: np.ndarray, active: np.ndarray | None = None) -> Stream:
    """Encode a residual stream as NVFP4 (see orc_encode_nvfp4). x, pred: uint16
    BF16 bits [T, H, D] (logical order); pred is the reconstruction X̂_{r-1}."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    pred = np.ascontiguousarray(pred, dtype=np.uint16)
    T, H, D = x.shape
    assert pred.shape == x.shape
    if active is not None:
        active = np.ascontiguousarray(active, dtype=np.int32)
        n = int(active.size)
    else:
        n = T
    codes = np.zeros((H, n, D // 2), dtype=np.uint8)
    bscale = np.zeros((H, n, D // 16), dtype=np.uint8)
    tscale = np.zeros(1, dtype=np.float32)
    rc = lib().orc_encode_nvfp4(kind, T, H, D, _ptr(x), _ptr(pred), _ptr(active), n, _ptr(codes), _ptr(bscale),
                                _ptr(tscale))
    if rc != 0:
        raise ValueError(f"orc_encode_nvfp4 failed with status {rc}")
    empty = np.zeros(0, dtype=np.uint16)
    return Stream(kind, T, H, D, n, active, codes, empty, empty, KGROUP_COMPACT, FMT_NVFP4, bscale, tscale)


def stream_bytes_nvfp4(n: int, H: int, D: int, sparse: bool = False) -> int:
    """Byte-exact payload of an NVFP4 stream: codes, E4M3 block scales, the FP32
    tensor scale (and the sparse index)."""
    return int(lib().orc_stream_bytes_nvfp4(n, H, D, int(sparse)))


def reconstruct(streams: list[Stream], depth: int, G: int = GROUP) -> np.ndarray:
    """BF16 bits [T, H, D] of the chain summed to `depth` (1 = base only)."""
    s0 = streams[0]
    arr = (_Stream * depth)(*[s.c_struct() for s in streams[:depth]])
    out = np.empty((s0.T, s0.H, s0.D), dtype=np.uint16)
    rc = lib().orc_reconstruct(s0.kind, s0.T, s0.H, s0.D, G, depth, arr, _ptr(out))
    if rc != 0:
        raise ValueError(f"orc_reconstruct failed with status {rc}")
    return out


def encode_chain(kind: int, xs: list[np.ndarray], actives: list[np.ndarray | None], G: int = GROUP,
                 kgroup: int = KGROUP_COMPACT, formats: list[int] | None = None) -> list[Stream]:
    """Loop 1 encodes X1 (INT4); loop r encodes X_r minus reconstruct(r-1) at its
    rows, in formats[r] (FMT_INT4 default, or FMT_NVFP4)."""
    streams = [encode(kind, xs[0], None, None, G, kgroup)]
    for r in range(1, len(xs)):
        pred = reconstruct(streams, r, G)
        if formats is not None and formats[r] == FMT_NVFP4:
            streams.append(encode_nvfp4(kind, xs[r], pred, actives[r]))
        else:
            streams.append(encode(kind, xs[r], pred, actives[r], G, kgroup))
    return streams


def attention(q: np.ndarray, khat: np.ndarray, vhat: np.ndarray, scale: float) -> np.ndarray:
    """FP32 decode attention of q [Hq, D] over K̂, V̂ [T, H, D] (all BF16 bits)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    khat = np.ascontiguousarray(khat, dtype=np.uint16)
    vhat = np.ascontiguousarray(vhat, dtype=np.uint16)
    Hq, D = q.shape
    T, H, D2 = khat.shape
    assert D2 == D and vhat.shape == khat.shape
    out = np.empty((Hq, D), dtype=np.float32)
    rc = lib().orc_attention(T, H, Hq, D, _ptr(q), _ptr(khat), _ptr(vhat), ctypes.c_float(scale), _ptr(out))
    if rc != 0:
        raise ValueError(f"orc_attention failed with status {rc}")
    return out


def stream_bytes(kind: int, n: int, H: int, D: int, G: int = GROUP, sparse: bool = False,
                 T: int | None = None, kgroup: int = KGROUP_COMPACT) -> int:
    """Byte-exact payload of one stream (codes, FP16 params, the sparse index)."""
    if T is None and kgroup == KGROUP_COMPACT:
        return int(lib().orc_stream_bytes(kind, n, H, D, G, int(sparse)))
    return int(lib().orc_stream_bytes_ex(kind, n, n if T is None else T, H, D, G, kgroup, int(sparse)))


def decode_f32(streams: list[Stream], depth: int, G: int = GROUP) -> np.ndarray:
    """FP32 [T, H, D] decode of the chain at `depth` with no BF16 rounding: the
    values a direct packed reader computes with (see orc_decode_f32)."""
    s0 = streams[0]
    arr = (_Stream * depth)(*[s.c_struct() for s in streams[:depth]])
    out = np.empty((s0.T, s0.H, s0.D), dtype=np.float32)
    rc = lib().orc_decode_f32(s0.kind, s0.T, s0.H, s0.D, G, depth, arr, _ptr(out))
    if rc != 0:
        raise ValueError(f"orc_decode_f32 failed with status {rc}")
    return out


def attention_f32(q: np.ndarray, kf: np.ndarray, vf: np.ndarray, scale: float) -> np.ndarray:
    """FP32 decode attention of q [Hq, D] (BF16 bits) over FP32 K, V [T, H, D]."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kf = np.ascontiguousarray(kf, dtype=np.float32)
    vf = np.ascontiguousarray(vf, dtype=np.float32)
    Hq, D = q.shape
    T, H, D2 = kf.shape
    assert D2 == D and vf.shape == kf.shape
    out = np.empty((Hq, D), dtype=np.float32)
    rc = lib().orc_attention_f32(T, H, Hq, D, _ptr(q), _ptr(kf), _ptr(vf), ctypes.c_float(scale), _ptr(out))
    if rc != 0:
        raise ValueError(f"orc_attention_f32 failed with status {rc}")
    return out


def attention_with_segments(q: np.ndarray, kf: np.ndarray, vf: np.ndarray, scale: float,
                            sink_k: np.ndarray | None = None, sink_v: np.ndarray | None = None,
                            tail_k: np.ndarray | None = None, tail_v: np.ndarray | None = None) -> np.ndarray:
    """FP32 decode attention over the FP32-decoded chain kf, vf [T, H, D] with the
    BF16 segments of a request (FlashLoop RFC §3.3 rolling BF16 tail; INT4 codec
    PR review, BF16 sink tokens): the first n_sink tokens take their BF16 values
    from sink_k / sink_v [n_sink, H, D] instead of the chain, and the tail tokens
    tail_k / tail_v [n_tail, H, D] follow the T chain tokens. BF16 as uint16 bits."""
    kf = np.array(kf, dtype=np.float32, copy=True)
    vf = np.array(vf, dtype=np.float32, copy=True)
    if sink_k is not None and len(sink_k):
        n = len(sink_k)
        kf[:n] = bf16_bits_to_f32(sink_k)
        vf[:n] = bf16_bits_to_f32(sink_v)
    if tail_k is not None and len(tail_k):
        kf = np.concatenate([kf, bf16_bits_to_f32(tail_k)], axis=0)
        vf = np.concatenate([vf, bf16_bits_to_f32(tail_v)], axis=0)
    if kf.shape[0] == 0:  # nothing to attend: zero output
        return np.zeros(np.asarray(q).shape, dtype=np.float32)
    return attention_f32(q, kf, vf, scale)


def request_path(xk: list[np.ndarray], xv: list[np.ndarray], actives: list[np.ndarray | None], q: np.ndarray,
                 depth: int, scale: float):
    """The whole path for one request: encode both chains, reconstruct to
    `depth` in BF16, and attend. Returns (k_streams, v_streams, khat, vhat,
    out) where `out` is the FP32 attention on the FP32 decode of the packed
    chains (the reference of the direct packed reader); the attention on the
    BF16 reconstruction is attention(q, khat, vhat, scale)."""
    ks = encode_chain(KIND_K, xk, actives)
    vs = encode_chain(KIND_V, xv, actives)
    khat = reconstruct(ks, depth)
    vhat = reconstruct(vs, depth)
    out = attention_f32(q, decode_f32(ks, depth), decode_f32(vs, depth), scale)
    return ks, vs, khat, vhat, out


# --------------------------------------------------------------------------- sparse decode attention


def sparse_reference(q: np.ndarray, kf: np.ndarray, vf: np.ndarray, scale: float, n_select: int):
    """Reference-loop state of sparse decode attention (FlashLoop RFC §3.2),
    in float64 from q [Hq, D] (BF16 bits) and the FP32 decode kf, vf [T, H, D]
    of the chain at the reference depth. Per query head h (KV head h // g):
      p      = softmax(q_h . k_t * scale) over all T keys
      S      = the n_select keys of largest p (equal p: lower position first),
               returned in ascending position order
      m      = sum of p over S
      O_ref  = sum_t p_t v_t        (the full attention output)
      C_ref  = sum over S of p_t v_t
    Returns (S [Hq, K] int32, m [Hq], O_ref [Hq, D], C_ref [Hq, D]), K = min(n_select, T)."""
    q64 = bf16_bits_to_f32(q).astype(np.float64)
    k64 = np.asarray(kf, dtype=np.float64)
    v64 = np.asarray(vf, dtype=np.float64)
    T, H, D = k64.shape
    Hq = q64.shape[0]
    g = Hq // H
    K = min(int(n_select), T)
    S = np.zeros((Hq, K), dtype=np.int32)
    m = np.zeros(Hq)
    o_ref = np.zeros((Hq, D))
    c_ref = np.zeros((Hq, D))
    for hq in range(Hq):
        h = hq // g
        s = k64[:, h, :] @ q64[hq] * scale
        p = np.exp(s - s.max())
        p /= p.sum()
        order = np.lexsort((np.arange(T), -p))  # largest p first, then lower position
        sel = np.sort(order[:K])
        S[hq] = sel
        m[hq] = p[sel].sum()
        o_ref[hq] = p @ v64[:, h, :]
        c_ref[hq] = p[sel] @ v64[sel, h, :]
    return S, m, o_ref, c_ref


def sparse_decode(q: np.ndarray, kf: np.ndarray, vf: np.ndarray, scale: float, S: np.ndarray, m: np.ndarray,
                  o_ref: np.ndarray, c_ref: np.ndarray) -> np.ndarray:
    """A later loop of sparse decode attention (FlashLoop RFC §3.2), float64:
      p_local = softmax(q_h . k_t * scale) over t in S (keys at this loop's depth)
      C_new   = m * sum over S of p_local_t v_t
      O       = O_ref - C_ref + C_new"""
    q64 = bf16_bits_to_f32(q).astype(np.float64)
    k64 = np.asarray(kf, dtype=np.float64)
    v64 = np.asarray(vf, dtype=np.float64)
    T, H, D = k64.shape
    Hq = q64.shape[0]
    g = Hq // H
    out = np.zeros((Hq, D))
    for hq in range(Hq):
        h = hq // g
        sel = np.asarray(S[hq], dtype=np.int64)
        if sel.size == 0:
            out[hq] = o_ref[hq] - c_ref[hq]
            continue
        s = k64[sel, h, :] @ q64[hq] * scale
        p = np.exp(s - s.max())
        p /= p.sum()
        out[hq] = o_ref[hq] - c_ref[hq] + m[hq] * (p @ v64[sel, h, :])
    return out
