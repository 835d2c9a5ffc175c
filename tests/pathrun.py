"""Runs one workload through the CUDA path (via the binding over the C ABI) and
through the CPU oracle, and compares them. Test-side helper: it is the one
place that sees both, and neither side imports the other."""

from __future__ import annotations

import json
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from oracle import oracle as O
from quantized_cross_loop_gb300 import kvq
from quantized_cross_loop_gb300.workloads import bf16_bits

from tests import reader_bound as RB

ATOL = 2e-3  # attention tolerance: |gpu - oracle| <= ATOL + RTOL * |oracle|
RTOL = 1e-2


def gpu_chains(req, device="cuda"):
    """Encode one request's K and V chains on the GPU. Returns (k_streams, v_streams)."""
    chains = []
    for kind, xs in ((kvq.KVQ_K, req.xk), (kvq.KVQ_V, req.xv)):
        s = [kvq.kvq_encode_base(xs[0].to(device), kind)]
        for r in range(1, len(xs)):
            act = req.active[r]
            s.append(kvq.kvq_encode_residual(xs[r].to(device), s, None if act is None else act.to(device)))
        chains.append(s)
    return chains[0], chains[1]


def gpu_attention(wl, k_chains, v_chains, depth, algo=kvq.ATTN_AUTO, q=None):
    table = kvq.RequestTable(k_chains, v_chains)
    q = (wl.q if q is None else q).to("cuda")
    ws = torch.empty(max(16, kvq.kvq_decode_attn_workspace_bytes(len(k_chains), wl.H, wl.Hq, wl.D)),
                     dtype=torch.uint8, device="cuda")
    out = kvq.kvq_decode_attn_packed(table, q, depth, wl.H, algo=algo, workspace=ws)
    torch.cuda.synchronize()
    return out, kvq.attn_error_word(ws)


def oracle_request(req, q_bits, depth, scale):
    xk = [bf16_bits(x) for x in req.xk]
    xv = [bf16_bits(x) for x in req.xv]
    act = [None if a is None else a.cpu().numpy().astype(np.int32) for a in req.active]
    return O.request_path(xk, xv, act, q_bits, depth, scale)


def oracle_many(reqs, q, depth, scale, threads=8):
    """Oracle results for several requests in parallel host threads (ctypes
    releases the GIL during each call)."""
    qb = bf16_bits(q)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda i: oracle_request(reqs[i], qb[i], depth, scale), range(len(reqs))))


def assert_stream_equal(gs, os_, what=""):
    """GPU stream planes equal the oracle's bit for bit."""
    codes = gs.codes_view().cpu().numpy()
    assert np.array_equal(codes, os_.codes), f"codes differ {what}: {np.argwhere(codes != os_.codes)[:5]}"
    mins = gs.mins_view().cpu().numpy().view(np.uint16)
    scales = gs.scales_view().cpu().numpy().view(np.uint16)
    assert np.array_equal(mins, os_.mins), f"mins differ {what}: {np.argwhere(mins != os_.mins)[:5]}"
    assert np.array_equal(scales, os_.scales), f"scales differ {what}"
    if os_.active is not None:
        assert np.array_equal(gs.active_view().cpu().numpy(), os_.active)


def assert_tile_dir(gs):
    if not gs.sparse:
        return
    act = gs.active_view().cpu().numpy()
    T = gs.n_tokens
    expect = np.searchsorted(act, np.arange(0, -(-T // 64) * 64 + 1, 64), side="left")
    assert np.array_equal(gs.tile_dir_view().cpu().numpy(), expect)


def assert_attention_close(out_gpu, out_ref, what=""):
    a = np.asarray(out_gpu, dtype=np.float64)
    b = np.asarray(out_ref, dtype=np.float64)
    err = np.abs(a - b)
    bound = ATOL + RTOL * np.abs(b)
    bad = err > bound
    assert not np.any(np.isnan(a)), f"NaN in GPU attention {what}"
    assert not bad.any(), (f"attention out of tolerance {what}: {bad.sum()} elements, max abs err "
                           f"{err.max():.3e}, worst at {np.unravel_index(np.argmax(err - bound), err.shape)}")
    return float(err.max()), float((err / np.maximum(np.abs(b), 1e-30)).max())


def accuracy_record(outs, refs):
    """Largest absolute error, largest relative error where |ref| >= 0.05, and
    the largest share of the per-element tolerance used, over a set of outputs."""
    a = np.concatenate([np.asarray(o, dtype=np.float64).ravel() for o in outs])
    b = np.concatenate([np.asarray(r, dtype=np.float64).ravel() for r in refs])
    err = np.abs(a - b)
    big = np.abs(b) >= 0.05
    return {"max_abs": float(err.max()),
            "max_rel_where_abs_ref_ge_0.05": float((err[big] / np.abs(b[big])).max()) if big.any() else None,
            "max_share_of_tolerance": float((err / (ATOL + RTOL * np.abs(b))).max())}


def log_accuracy(what, outs, refs):
    """Appends accuracy_record(outs, refs) as one JSON line to the file named by
    KVQ_ACCURACY_LOG, when that variable is set (a record of the attention
    error per configuration beside the pass/fail check)."""
    path = os.environ.get("KVQ_ACCURACY_LOG")
    if not path:
        return
    rec = {"case": what, **accuracy_record(outs, refs)}
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def assert_reader_error_bounded(out_gpu, o_ref, ks, vs, khat, vhat, q_bits, depth, scale, what=""):
    """The GPU attention against the attention over the BF16 reconstruction
    X̂: |gpu - o(X̂)| <= |gpu - o(X̃)| + |o(X̃) - o(X̂)|, the first within the
    attention tolerance of o(X̃) = o_ref, the second within the direct-reader
    bound derived in tests/reader_bound.py (FlashLoop RFC §9 asks that error
    bounded). Returns the largest |gpu - o(X̂)| and the bound there."""
    o_bf = O.attention(q_bits, khat, vhat, scale).astype(np.float64)
    bound = RB.reader_error_bound(q_bits, ks, vs, depth, scale)
    gap = np.abs(o_bf - np.asarray(o_ref, dtype=np.float64))
    assert np.all(gap <= bound), f"oracle direct-reader gap {gap.max():.3e} above its bound {what}"
    err = np.abs(np.asarray(out_gpu, dtype=np.float64) - o_bf)
    lim = ATOL + RTOL * np.abs(np.asarray(o_ref, dtype=np.float64)) + bound
    assert np.all(err <= lim), f"direct-reader error {err.max():.3e} above its derived bound {what}"
    k = int(np.argmax(err))
    return float(err.flat[k]), float(lim.flat[k])


def softmax_scale(D):
    return 1.0 / math.sqrt(D)
