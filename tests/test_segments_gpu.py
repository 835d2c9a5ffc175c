"""Packed decode attention with the BF16 segments of a request, through the C ABI,
against the oracle on the same data: the first n_sink tokens read from a BF16
sink instead of the packed chain, n_tail BF16 tokens after the packed ones
(FlashLoop RFC, vllm-rlt issue #156, §3.3 rolling BF16 tail; INT4 codec PR,
vllm-rlt pull #166, review: BF16 sink and recent window)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_cross_loop_gb300 import kvq
from quantized_cross_loop_gb300 import workloads as W
from quantized_cross_loop_gb300.workloads import bf16_bits

from tests import pathrun as P

pytestmark = pytest.mark.gpu

ALGOS = [kvq.ATTN_SIMT, kvq.ATTN_MMA, kvq.ATTN_MMA_GENERAL, kvq.ATTN_TCGEN05]
H, D = 8, 128


def _request(T, sparse, seed):
    spec = W.ConfigSpec("seg", seed, 1, max(T, 1), H, D, 32, 4, 0.1,
                        (1.0, 1.0, 0.5, 0.25) if sparse else (1.0, 1.0, 1.0, 1.0))
    return W.make_request(spec, 0, 0, "cpu", T=T, sparse=sparse)


def _segments(ns, nt, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda n: torch.randn((n, H, D), generator=g).to(torch.bfloat16)  # noqa: E731
    return mk(ns), mk(ns), mk(nt), mk(nt)


def _oracle(req, q_bits, seg, depth=4):
    scale = P.softmax_scale(D)
    if req.T > 0:
        xk = [bf16_bits(x) for x in req.xk]
        xv = [bf16_bits(x) for x in req.xv]
        act = [None if a is None else a.numpy().astype(np.int32) for a in req.active]
        kf = O.decode_f32(O.encode_chain(O.KIND_K, xk, act), depth)
        vf = O.decode_f32(O.encode_chain(O.KIND_V, xv, act), depth)
    else:
        kf = vf = np.zeros((0, H, D), dtype=np.float32)
    sk, sv, tk, tv = (bf16_bits(t) for t in seg)
    return O.attention_with_segments(q_bits, kf, vf, scale, sk, sv, tk, tv)


def _run(reqs, segs, Hq=32):
    kc, vc = [], []
    for r in reqs:
        k, v = P.gpu_chains(r)
        kc.append(k)
        vc.append(v)
    dsegs = [None if s is None else tuple(t.cuda() for t in s) for s in segs]
    table = kvq.RequestTable(kc, vc, torch.device("cuda"), segments=dsegs)
    q = torch.randn((len(reqs), Hq, D), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    outs = {}
    for algo in ALGOS:
        ws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(len(reqs), H, Hq, D), dtype=torch.uint8, device="cuda")
        out = kvq.kvq_decode_attn_packed(table, q.cuda(), 4, H, algo=algo, workspace=ws)
        torch.cuda.synchronize()
        outs[algo] = (out.cpu().numpy(), kvq.attn_error_word(ws))
    return q, outs


@pytest.mark.parametrize("T,sparse,ns,nt", [
    (1000, True, 4, 100),   # sink of 4, partial last tile, sparse loops, tail
    (256, False, 64, 64),   # the sink covers the first tile exactly
    (300, True, 300, 0),    # every packed token replaced by the sink
    (0, False, 0, 127),     # nothing packed yet: the tail alone
    (130, False, 0, 1),     # one tail token
    (70, True, 5, 0),       # sink only
])
def test_segments_single_request(T, sparse, ns, nt):
    req = _request(T, sparse, 40 + T + ns)
    seg = _segments(ns, nt, 7 + nt)
    q, outs = _run([req], [seg])
    ref = _oracle(req, bf16_bits(q[0]), seg)
    for algo, (out, err) in outs.items():
        assert err == 0
        P.assert_attention_close(out[0], ref, f"T {T} sink {ns} tail {nt} algo {algo}")


def test_segments_mixed_batch_with_split_units():
    """Requests with and without segments in one call; long requests are split
    over several blocks (their partials merge before the segments do)."""
    reqs = [_request(4096, False, 51), _request(1000, True, 52), _request(200, False, 53), _request(3000, True, 54)]
    segs = [_segments(4, 127, 1), None, _segments(0, 64, 2), _segments(16, 0, 3)]
    q, outs = _run(reqs, segs)
    none = tuple(torch.zeros((0, H, D), dtype=torch.bfloat16) for _ in range(4))
    for b, r in enumerate(reqs):
        ref = _oracle(r, bf16_bits(q[b]), segs[b] if segs[b] is not None else none)
        for algo, (out, err) in outs.items():
            assert err == 0
            P.assert_attention_close(out[b], ref, f"req {b} algo {algo}")


def test_segments_inconsistent_entry_is_flagged():
    """A sink longer than the packed tokens: that request's output is NaN and
    the error word is set; the other request is unaffected."""
    reqs = [_request(100, False, 61), _request(100, False, 62)]
    segs = [_segments(101, 0, 4), None]
    q, outs = _run(reqs, segs)
    none = tuple(torch.zeros((0, H, D), dtype=torch.bfloat16) for _ in range(4))
    ref1 = _oracle(reqs[1], bf16_bits(q[1]), none)
    for algo, (out, err) in outs.items():
        assert err != 0
        assert np.all(np.isnan(out[0]))
        P.assert_attention_close(out[1], ref1, f"algo {algo}")


def test_segments_many_units_grid_stride():
    """More (request, KV head) units than the epilogue kernels' grid (two blocks
    per attention CTA): requests with segments far apart in the table, empty
    requests with and without a tail, short packed requests, all in one call."""
    n = 90  # 720 units
    reqs, segs = [], []
    for b in range(n):
        T = (0, 64, 1, 130)[b % 4]
        reqs.append(_request(T, T > 64 and b % 3 == 0, 300 + b))
        segs.append(_segments(min(2, T), 5, 900 + b) if b in (1, 42, 44, 83, 87, 89) else None)
    q, outs = _run(reqs, segs)
    none = tuple(torch.zeros((0, H, D), dtype=torch.bfloat16) for _ in range(4))
    for b, r in enumerate(reqs):
        ref = _oracle(r, bf16_bits(q[b]), segs[b] if segs[b] is not None else none)
        for algo, (out, err) in outs.items():
            assert err == 0
            P.assert_attention_close(out[b], ref, f"req {b} algo {algo}")
