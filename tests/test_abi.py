"""The C ABI without a GPU: libkvq.so builds for sm_103a, loads, exports every
function include/kvq.h declares, and rejects bad arguments on the host before
any launch. No compute call is made here."""

from __future__ import annotations

import ctypes
import os
import re

import pytest

from quantized_cross_loop_gb300 import build as kbuild
from quantized_cross_loop_gb300 import kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kvq.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("kvq_encode_base", "kvq_encode_residual", "kvq_reconstruct", "kvq_decode_attn_packed"):
        assert n in names
    assert set(names) == set(kvq.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {kvq.LIB_PATH}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", out), name


def test_library_is_built_for_sm_103a(L):
    out = os.popen(f"cuobjdump --list-elf {kvq.LIB_PATH} 2>&1").read()
    assert "sm_103a" in out, out


def test_struct_layouts_match_header():
    src = r'''
#include <stdio.h>
#include <stddef.h>
#include "kvq.h"
int main(void){printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(kvq_stream), offsetof(kvq_stream, codes),
  offsetof(kvq_stream, tile_dir), sizeof(kvq_loop_ref), sizeof(kvq_request), offsetof(kvq_request, n_sink),
  offsetof(kvq_request, tail_v), offsetof(kvq_stream, kgroup), offsetof(kvq_loop_ref, flags),
  offsetof(kvq_stream, format), offsetof(kvq_stream, token_cap), offsetof(kvq_loop_ref, kgroup_cap)); return 0;}
'''
    import subprocess
    import tempfile

    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "s.c")
        open(c, "w").write(src)
        exe = os.path.join(d, "s")
        subprocess.run(["gcc", "-I" + os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        got = [int(v) for v in subprocess.run([exe], capture_output=True, text=True).stdout.split()]
    assert got == [ctypes.sizeof(kvq.kvq_stream), kvq.kvq_stream.codes.offset, kvq.kvq_stream.tile_dir.offset,
                   ctypes.sizeof(kvq.kvq_loop_ref), ctypes.sizeof(kvq.kvq_request), kvq.kvq_request.n_sink.offset,
                   kvq.kvq_request.tail_v.offset, kvq.kvq_stream.kgroup.offset, kvq.kvq_loop_ref.flags.offset,
                   kvq.kvq_stream.format.offset, kvq.kvq_stream.token_cap.offset, kvq.kvq_loop_ref.kgroup_cap.offset]


def test_plane_sizes_and_payload(L):
    from oracle import oracle as O

    for kind in (kvq.KVQ_K, kvq.KVQ_V):
        for n, T in ((0, 10), (1, 1), (65, 100), (500, 1000), (4096, 4096)):
            s = kvq.kvq_stream()
            assert L.kvq_stream_init(ctypes.byref(s), kind, n, T, 8, 128) == 0
            sizes = [L.kvq_plane_bytes(ctypes.byref(s), p) for p in range(5)]
            assert all(v % 16 == 0 for v in sizes)
            assert sizes[0] >= 8 * n * 64
            assert sizes[3] >= 16 and sizes[4] >= 4 * (-(-T // 64) + 1)
            for sparse in (0, 1):
                # byte-exact storage agrees with the oracle's own accounting
                assert L.kvq_stream_payload_bytes(kind, n, 8, 128, sparse) == O.stream_bytes(kind, n, 8, 128,
                                                                                               sparse=bool(sparse))
                # and under tile grouping of K (ceil(T/64) groups of a sparse stream)
                assert L.kvq_stream_payload_bytes_ex(kind, n, T, 8, 128, sparse, kvq.KVQ_KGROUP_TILE,
                                                     kvq.KVQ_FMT_INT4) == \
                    O.stream_bytes(kind, n, 8, 128, sparse=bool(sparse), T=T, kgroup=O.KGROUP_TILE)
                # and for an NVFP4 residual stream
                assert L.kvq_stream_payload_bytes_ex(kind, n, T, 8, 128, sparse, kvq.KVQ_KGROUP_COMPACT,
                                                     kvq.KVQ_FMT_NVFP4) == O.stream_bytes_nvfp4(n, 8, 128, bool(sparse))
            nv = kvq.kvq_stream()
            assert L.kvq_stream_init(ctypes.byref(nv), kind, n, T, 8, 128) == 0
            assert L.kvq_stream_set_format(ctypes.byref(nv), kvq.KVQ_FMT_NVFP4) == 0 and nv.group == 16
            assert L.kvq_plane_bytes(ctypes.byref(nv), 1) == -(-(8 * n * 8) // 16) * 16  # E4M3 per 16 channels
            assert L.kvq_plane_bytes(ctypes.byref(nv), 2) == 16                          # tensor-scale record
            assert L.kvq_stream_set_format(ctypes.byref(nv), 7) == -1
            s.kgroup = kvq.KVQ_KGROUP_TILE
            groups = (-(-T // 64) if n > 0 else 0) if kind == kvq.KVQ_K else None
            if groups is not None:
                assert L.kvq_plane_bytes(ctypes.byref(s), 1) == -(-(2 * 8 * groups * 128) // 16) * 16


def _stream(L, kind=0, n=64, T=64, H=8, D=128):
    s = kvq.kvq_stream()
    L.kvq_stream_init(ctypes.byref(s), kind, n, T, H, D)
    return s


def test_host_validation_rejects_bad_arguments(L):
    """Each call returns an error status before touching the device."""
    BAD, UNSUP, MIS = -1, -2, -3
    s = _stream(L)
    assert L.kvq_encode_base(None, None, None) == BAD
    assert b"NULL" in L.kvq_last_error()
    s.codes, s.mins, s.scales = 16, 32, 48
    s.version = 7
    assert L.kvq_encode_base(ctypes.c_void_p(64), ctypes.byref(s), None) == UNSUP
    s.version = 1
    s.head_dim = 64
    assert L.kvq_encode_base(ctypes.c_void_p(64), ctypes.byref(s), None) == UNSUP
    s.head_dim = 128
    s.codes = 17  # misaligned
    assert L.kvq_encode_base(ctypes.c_void_p(64), ctypes.byref(s), None) == MIS
    s.codes = 16
    s.n_rows = 10  # dense stream whose rows differ from its tokens
    assert L.kvq_encode_base(ctypes.c_void_p(64), ctypes.byref(s), None) == BAD
    # residual: the base of the chain must be dense, depth within bounds
    prev = (kvq.kvq_stream * 1)(_stream(L))
    prev[0].codes, prev[0].mins, prev[0].scales = 16, 32, 48
    out = _stream(L)
    out.codes, out.mins, out.scales = 16, 32, 48
    assert L.kvq_encode_residual(ctypes.c_void_p(64), prev, 0, ctypes.byref(out), None) == BAD
    assert L.kvq_encode_residual(ctypes.c_void_p(64), prev, 8, ctypes.byref(out), None) == BAD
    prev[0].active_idx = 64
    prev[0].n_rows = 32
    prev[0].tile_dir = 64
    assert L.kvq_encode_residual(ctypes.c_void_p(64), prev, 1, ctypes.byref(out), None) == BAD
    # sparse output without tile_dir storage
    prev[0].active_idx, prev[0].n_rows, prev[0].tile_dir = None, 64, None
    out.active_idx, out.n_rows = 64, 32
    assert L.kvq_encode_residual(ctypes.c_void_p(64), prev, 1, ctypes.byref(out), None) == BAD
    # NVFP4 is a residual format: the base refuses it, and so does a chain whose base carries it
    out.active_idx, out.n_rows = None, 64
    nv = _stream(L)
    nv.codes, nv.mins, nv.scales = 16, 32, 48
    assert L.kvq_stream_set_format(ctypes.byref(nv), kvq.KVQ_FMT_NVFP4) == 0
    assert L.kvq_encode_base(ctypes.c_void_p(64), ctypes.byref(nv), None) == UNSUP
    nvprev = (kvq.kvq_stream * 1)(nv)
    assert L.kvq_encode_residual(ctypes.c_void_p(64), nvprev, 1, ctypes.byref(out), None) == UNSUP
    nv.group = 64  # NVFP4 with the INT4 group size: not a format the kernels read
    assert L.kvq_encode_residual(ctypes.c_void_p(64), prev, 1, ctypes.byref(nv), None) == UNSUP
    # batched calls: the base bit of the NVFP4 loop mask must be clear
    ws = ctypes.create_string_buffer(64)
    assert L.kvq_encode_batch_ex(ctypes.c_void_p(64), 1, 8, 128, 0, 1, ctypes.c_void_p(64), 1, ws, 64, None) == BAD
    assert b"nvfp4_loops" in L.kvq_last_error()
    assert L.kvq_reconstruct_batch_ex(ctypes.c_void_p(64), 1, 8, 128, 0, 2, ctypes.c_void_p(64), 1, ws, 64,
                                      None) == BAD
    # attention: shape checks come first
    f = L.kvq_decode_attn_packed_ex
    assert f(None, 1, 8, 30, 128, 4, None, ctypes.c_float(0.1), None, None, 0, 0, None) == BAD  # 30 % 8
    assert f(None, 1, 8, 96, 128, 4, None, ctypes.c_float(0.1), None, None, 0, 0, None) == UNSUP  # g = 12
    assert f(None, 1, 8, 32, 64, 4, None, ctypes.c_float(0.1), None, None, 0, 0, None) == UNSUP
    assert f(None, 1, 8, 32, 128, 0, None, ctypes.c_float(0.1), None, None, 0, 0, None) == BAD
    assert f(None, 1, 8, 32, 128, 9, None, ctypes.c_float(0.1), None, None, 0, 0, None) == BAD
    assert f(None, 1, 8, 32, 128, 4, None, ctypes.c_float(-1.0), None, None, 0, 0, None) == BAD
    assert f(None, 1, 8, 32, 128, 4, None, ctypes.c_float(0.1), None, None, 0, 5, None) == BAD
    assert f(None, 1, 8, 32, 128, 4, None, ctypes.c_float(0.1), None, None, 0, 0, None) == BAD  # NULL pointers
    assert L.kvq_status_string(-4) == b"KVQ_ERR_WORKSPACE"
    # sparse later loop: algo, then the workspace the chosen kernel needs (no device work before either)
    sp = L.kvq_sparse_decode_attn_ex
    p16, ws16 = ctypes.c_void_p(64), ctypes.create_string_buffer(32)
    ws_al = ctypes.c_void_p((ctypes.addressof(ws16) + 15) // 16 * 16)
    args = (p16, 1, 8, 32, 128, 4, p16, ctypes.c_float(0.1), 4, 64, p16, p16, p16, p16, p16)
    assert sp(*args, ws_al, 16, 5, None) == BAD  # not an algo
    assert sp(*args, ws_al, 8, 0, None) == -4  # below the 16 bytes of the error word
    assert sp(*args, ws_al, 16, 2, None) in (-4, -5)  # the tensor-core path asked for with 16 bytes (or no GPU here)
    assert L.kvq_sparse_decode_workspace_bytes(-1, 8, 32, 128, 64) == 0
    assert L.kvq_sparse_decode_workspace_bytes(1, 0, 32, 128, 64) == 0


def test_request_fill_checks_pairs(L):
    k = (kvq.kvq_stream * 2)(_stream(L, 0), _stream(L, 0, n=32))
    v = (kvq.kvq_stream * 2)(_stream(L, 1), _stream(L, 1, n=32))
    for arr in (k, v):
        for s in arr:
            s.codes, s.mins, s.scales = 16, 32, 48
        arr[1].active_idx, arr[1].tile_dir = 64, 80
    req = kvq.kvq_request()
    assert L.kvq_request_fill(k, v, 2, ctypes.byref(req)) == 0
    assert req.n_tokens == 64 and req.n_loops == 2 and req.loop[1].n_rows == 32 and req.loop[1].tile_dir == 80
    v[1].n_rows = 31
    assert L.kvq_request_fill(k, v, 2, ctypes.byref(req)) == -1
    v[1].n_rows = 32
    assert L.kvq_request_fill(v, k, 2, ctypes.byref(req)) == -1  # kinds swapped
