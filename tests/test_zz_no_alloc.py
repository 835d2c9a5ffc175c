"""The allocation-free decode attention entry point.

Callers that cannot allocate device memory (code under CUDA graph capture,
plugins inside a serving process that owns every allocation) call
kvq_decode_attn_packed_noalloc, which uses the library's static device scratch
instead of a caller workspace. It runs the same plan and kernels as the
workspace entry point, so its output must equal that entry point's bit for bit,
on two calls in a row and after a smaller call; it must allocate nothing; a
request it refuses shows as NaN rows (its error word lives in the static
scratch, out of the caller's reach); sizes beyond the static scratch are
refused before any launch. This file is collected last.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from quantized_cross_loop_gb300 import kvq
from quantized_cross_loop_gb300 import workloads as W

from tests import pathrun as P

pytestmark = pytest.mark.gpu


def _batch():
    spec = W.CONFIGS[2]
    reqs = [W.make_request(spec, 0, b, "cuda") for b in range(3)]
    reqs.append(W.make_request(spec, 0, 7, "cuda", T=333, sparse=False))
    k, v = [], []
    for r in reqs:
        kc, vc = P.gpu_chains(r)
        k.append(kc)
        v.append(vc)
    table = kvq.RequestTable(k, v)
    q = W.make_queries(spec, 0, len(reqs), "cuda")
    return table, q


def _same(a: np.ndarray, b: np.ndarray) -> bool:
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_noalloc_matches_workspace_entry_point_twice():
    table, q = _batch()
    ref = kvq.kvq_decode_attn_packed(table, q, 4, 8).cpu().numpy()
    out = torch.empty_like(torch.from_numpy(ref)).cuda()
    kvq.kvq_decode_attn_packed_noalloc(table, q, 4, 8, out=out)  # loads the module and its scratch
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        out.fill_(float("nan"))
        kvq.kvq_decode_attn_packed_noalloc(table, q, 4, 8, out=out)
        torch.cuda.synchronize()
        assert _same(out.cpu().numpy(), ref), "noalloc differs from the workspace entry point"
    assert torch.cuda.mem_get_info()[0] == free0, "the no-alloc entry point allocated device memory"
    # a smaller call in between must not see stale partials of the larger one
    sub = kvq.RequestTable(table._keep[0][:1], table._keep[1][:1])
    got1 = kvq.kvq_decode_attn_packed_noalloc(sub, q[:1].contiguous(), 3, 8).cpu().numpy()
    ref1 = kvq.kvq_decode_attn_packed(sub, q[:1].contiguous(), 3, 8).cpu().numpy()
    assert _same(got1, ref1), "noalloc, one request at depth 3"
    got = kvq.kvq_decode_attn_packed_noalloc(table, q, 4, 8).cpu().numpy()
    assert _same(got, ref), "noalloc after a smaller call"


def test_noalloc_refuses_nvfp4_requests_with_nan_rows():
    """The no-alloc entry reads INT4 tables: a request holding NVFP4 loops is
    refused on the device (NaN rows, as the workspace entry point without the
    NVFP4 flag does); the INT4 request beside it is unaffected."""
    from tests.test_nvfp4_gpu import _nvfp4_requests

    H, Hq, D = 8, 32, 128
    _, kc, vc, _, _, _ = _nvfp4_requests([300], Hq, 700)
    _, kc4, vc4, _, _, _ = _nvfp4_requests([200], Hq, 701, (kvq.KVQ_FMT_INT4,) * 4)
    table = kvq.RequestTable(kc + kc4, vc + vc4, torch.device("cuda"))
    q = torch.randn((2, Hq, D), generator=torch.Generator().manual_seed(702)).to(torch.bfloat16).cuda()
    ws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(2, H, Hq, D), dtype=torch.uint8, device="cuda")
    ref = torch.empty((2, Hq, D), dtype=torch.float32, device="cuda")
    L = kvq.lib()
    st = L.kvq_decode_attn_packed_ex(kvq._dptr(table.table), 2, H, Hq, D, 4, kvq._dptr(q), ctypes.c_float(0.088),
                                     kvq._dptr(ref), kvq._dptr(ws), ws.numel(), kvq.ATTN_AUTO, None)
    assert st == 0
    got = kvq.kvq_decode_attn_packed_noalloc(table, q, 4, H, softmax_scale=0.088)
    torch.cuda.synchronize()
    g, r = got.cpu().numpy(), ref.cpu().numpy()
    assert kvq.attn_error_word(ws) & 64
    assert np.all(np.isnan(g[0])) and np.all(np.isnan(r[0]))
    assert _same(g[1], r[1])


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    L = kvq.lib()
    f = L.kvq_decode_attn_packed_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int32
    # 100000 requests x 8 heads needs far more than 32 MiB; refused before any launch
    st = f(ctypes.c_void_p(256), 100000, 8, 32, 128, 4, ctypes.c_void_p(256), ctypes.c_float(0.088),
           ctypes.c_void_p(256), None)
    assert st == -4
    assert b"static scratch" in L.kvq_last_error()
