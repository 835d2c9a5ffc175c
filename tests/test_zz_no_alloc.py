"""The allocation-free decode attention entry point.

Callers that cannot allocate device memory (code under CUDA graph capture,
plugins inside a serving process that owns every allocation) call
kvq_decode_attn_packed_noalloc, which uses the library's static device scratch
instead of a caller workspace. Its output must match the workspace entry point
within the attention tolerance on two calls in a row, and sizes beyond the
static scratch must be refused before any launch. This file is collected last.
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


def test_noalloc_matches_workspace_entry_point_twice():
    table, q = _batch()
    ref = kvq.kvq_decode_attn_packed(table, q, 4, 8).cpu().numpy()
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        got = kvq.kvq_decode_attn_packed_noalloc(table, q, 4, 8)
        torch.cuda.synchronize()
        P.assert_attention_close(got.cpu().numpy(), ref, "noalloc vs workspace entry point")
    # a smaller call in between must not see stale partials of the larger one
    sub = kvq.RequestTable(table._keep[0][:1], table._keep[1][:1])
    got1 = kvq.kvq_decode_attn_packed_noalloc(sub, q[:1].contiguous(), 3, 8).cpu().numpy()
    ref1 = kvq.kvq_decode_attn_packed(sub, q[:1].contiguous(), 3, 8).cpu().numpy()
    P.assert_attention_close(got1, ref1, "noalloc, one request at depth 3")


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
