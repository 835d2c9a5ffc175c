"""CUDA path vs CPU oracle, element by element, through the C ABI.

Codec planes (codes, FP16 mins/scales), tile directories and reconstructions
must be bit-exact; decode attention must satisfy |gpu - oracle| <= 2e-3 +
1e-2 * |oracle| per element (FP32 oracle on the same packed data)."""

from __future__ import annotations

import os

import numpy as np
import pytest
import torch

from quantized_cross_loop_gb300 import kvq
from quantized_cross_loop_gb300 import workloads as W
from quantized_cross_loop_gb300.workloads import bf16_bits

from tests import pathrun as P

pytestmark = pytest.mark.gpu

ALGOS = [kvq.ATTN_SIMT, kvq.ATTN_MMA, kvq.ATTN_MMA_GENERAL, kvq.ATTN_TCGEN05]
THREADS = max(1, min(16, os.cpu_count() or 1))


def _algos():
    return ALGOS


def check_workload(wl, sample=None, depths=(4,), full_recon=True):
    """Encode every request on the GPU, attend at each depth; compare the
    sampled requests (default: all) with the oracle."""
    kc, vc = [], []
    for req in wl.requests:
        k, v = P.gpu_chains(req)
        kc.append(k)
        vc.append(v)
    sample = list(range(wl.n_requests)) if sample is None else list(sample)
    scale = P.softmax_scale(wl.D)
    for depth in depths:
        ref = P.oracle_many([wl.requests[i] for i in sample], wl.q[sample].cpu(), depth, scale, THREADS)
        for algo in _algos():
            out, err = P.gpu_attention(wl, kc, vc, depth, algo)
            assert err == 0
            out = out.cpu().numpy()
            P.log_accuracy(f"{wl.spec.name} layer {wl.layer} x{wl.n_requests} depth {depth} algo {algo} "
                           f"({len(sample)} requests)", [out[i] for i in sample],
                           [r[4] for r in ref])
            for j, i in enumerate(sample):
                ks, vs, khat, vhat, o_ref = ref[j]
                if depth == depths[0] and algo == _algos()[0]:
                    for r in range(wl.depth):
                        P.assert_stream_equal(kc[i][r], ks[r], f"K req {i} loop {r + 1}")
                        P.assert_stream_equal(vc[i][r], vs[r], f"V req {i} loop {r + 1}")
                        P.assert_tile_dir(kc[i][r])
                    if full_recon:
                        rk = kvq.kvq_reconstruct(kc[i], depth)
                        rv = kvq.kvq_reconstruct(vc[i], depth)
                        assert np.array_equal(bf16_bits(rk), khat), f"K reconstruct req {i}"
                        assert np.array_equal(bf16_bits(rv), vhat), f"V reconstruct req {i}"
                P.assert_attention_close(out[i], o_ref, f"req {i} depth {depth} algo {algo}")
                P.assert_reader_error_bounded(out[i], o_ref, ks, vs, khat, vhat, bf16_bits(wl.q[i]), depth, scale,
                                              f"req {i} depth {depth} algo {algo}")
    return kc, vc


@pytest.mark.parametrize("cfg", [1, 2])
def test_small_configs_full(cfg):
    wl = W.make_workload(cfg, device="cpu")
    check_workload(wl, depths=(1, 2, 3, 4))


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 129, 200])
def test_edge_lengths(T):
    spec = W.ConfigSpec("edge", 50 + T, 1, T, 8, 128, 32, 4, 0.1, (1.0, 1.0, 0.5, 0.25))
    reqs = [W.make_request(spec, 0, 0, "cpu")]
    q = W.make_queries(spec, 0, 1)
    wl = W.Workload(spec, 0, 8, 128, 32, 4, reqs, q)
    check_workload(wl, depths=(1, 4))


@pytest.mark.parametrize("H,Hq", [(1, 1), (3, 6), (2, 16), (8, 64)])
def test_head_layouts(H, Hq):
    spec = W.ConfigSpec("heads", 70 + H, 2, 150, H, 128, Hq, 4, 0.1, (1.0, 1.0, 0.5, 0.25))
    reqs = [W.make_request(spec, 0, b, "cpu") for b in range(2)]
    wl = W.Workload(spec, 0, H, 128, Hq, 4, reqs, W.make_queries(spec, 0, 2))
    check_workload(wl, depths=(4,))


def test_special_active_sets():
    """Empty, single and full sparse sets; sets that straddle K groups and tiles."""
    T, H = 300, 8
    spec = W.ConfigSpec("sets", 90, 1, T, H, 128, 32, 4, 0.1, (1.0, 1.0, 1.0, 1.0))
    base = W.make_request(spec, 0, 0, "cpu")
    cases = [
        (torch.arange(T, dtype=torch.int32), torch.arange(0, T, 2, dtype=torch.int32)),  # full, then half
        (torch.tensor([5], dtype=torch.int32), torch.tensor([], dtype=torch.int32)),  # single, then empty
        (torch.arange(60, 200, dtype=torch.int32), torch.arange(63, 130, dtype=torch.int32)),  # straddles
        (torch.tensor([0, 63, 64, 127, 128, 299], dtype=torch.int32), torch.tensor([63, 64, 299], dtype=torch.int32)),
    ]
    reqs = [W.Request(T, base.xk, base.xv, [None, None, a3, a4]) for a3, a4 in cases]
    wl = W.Workload(spec, 0, H, 128, 32, 4, reqs, W.make_queries(spec, 0, len(reqs)))
    check_workload(wl, depths=(2, 3, 4))


def test_batched_ragged_with_empty_request():
    spec = W.ConfigSpec("ragged", 91, 5, None, 8, 128, 32, 4, 0.1, (1.0, 1.0, 0.5, 0.25))
    lengths = [0, 1, 700, 64, 1337]
    reqs = [W.make_request(spec, 0, b, "cpu", T=t, sparse=(b % 2 == 1)) for b, t in enumerate(lengths)]
    wl = W.Workload(spec, 0, 8, 128, 32, 4, reqs, W.make_queries(spec, 0, len(reqs)))
    kc, vc = [], []
    for req in reqs:
        k, v = P.gpu_chains(req)
        kc.append(k)
        vc.append(v)
    for algo in _algos():
        out, err = P.gpu_attention(wl, kc, vc, 4, algo)
        assert err == 0
        out = out.cpu().numpy()
        assert np.all(out[0] == 0.0)  # no stored tokens: zero output
        ref = P.oracle_many(reqs[1:], wl.q[1:].cpu(), 4, P.softmax_scale(128), THREADS)
        for j in range(1, len(reqs)):
            P.assert_attention_close(out[j], ref[j - 1][4], f"req {j} algo {algo}")


@pytest.mark.parametrize("cfg,sample", [(3, [0, 31]), (4, [2])])
def test_large_configs_sampled(cfg, sample):
    """Full-size workload on the GPU (device-generated inputs, the bench's launch
    configuration); the oracle checks the sampled requests end to end."""
    wl = W.make_workload(cfg, device="cuda")
    check_workload(wl, sample=sample, depths=(4,), full_recon=True)


def test_replicated_partial_sparse_sampled():
    """512 independent copies of the partial-group sparse configuration in one
    batched call; the oracle checks a few of them."""
    wl = W.make_workload(2, device="cuda", replicate=512)
    check_workload(wl, sample=[0, 257, 511], depths=(4,))


@pytest.mark.parametrize("layer", [0, 23])
def test_ragged_layers_sampled(layer):
    """The ragged multi-layer sweep: one layer, all 64 requests on the GPU; the
    oracle checks one dense and one sparse request."""
    wl = W.make_workload(5, device="cuda", layer=layer)
    sp = W.request_is_sparse(wl.spec)
    sample = [sp.index(False), sp.index(True)]
    check_workload(wl, sample=sample, depths=(4,), full_recon=False)


def test_attention_error_word_for_bad_table():
    """A request whose table entry is inconsistent (depth beyond its loops)
    gets NaN output and sets the error word; the others are unaffected."""
    spec = W.CONFIGS[1]
    reqs = [W.make_request(spec, 0, 0, "cpu")]
    k, v = P.gpu_chains(reqs[0])
    table = kvq.RequestTable([k[:2], k[:2]], [v[:2], v[:2]])
    raw = table.table.view(-1)
    # the second entry claims only one stored loop
    off = kvq.ctypes.sizeof(kvq.kvq_request)
    raw[off + 4:off + 8] = torch.tensor([1, 0, 0, 0], dtype=torch.uint8)
    q = W.make_queries(spec, 0, 2).cuda()
    ws = torch.zeros(kvq.kvq_decode_attn_workspace_bytes(2, 8, 32, 128), dtype=torch.uint8, device="cuda")
    for algo in _algos():
        out = kvq.kvq_decode_attn_packed(table, q, 2, 8, algo=algo, workspace=ws)
        torch.cuda.synchronize()
        assert kvq.attn_error_word(ws) != 0
        o = out.cpu().numpy()
        assert np.all(np.isnan(o[1])) and not np.any(np.isnan(o[0]))


def test_batch_api_matches_single_request_api():
    """The batched encode and reconstruction (device request table, one pool of
    contiguous per-request planes) give the same bytes as the per-request calls,
    and the attention over the pool matches the oracle."""
    spec = W.CONFIGS[2]
    reqs = [W.make_request(spec, 0, b, "cpu") for b in range(3)]
    reqs += [W.make_request(W.CONFIGS[1], 0, 0, "cpu")]
    reqs += [W.make_request(spec, 0, 9, "cpu", T=1, sparse=True), W.make_request(spec, 0, 10, "cpu", T=0)]
    dev = torch.device("cuda")
    dreqs = [W.Request(r.T, [x.to(dev) for x in r.xk], [x.to(dev) for x in r.xv],
                       [None if a is None else a.to(dev) for a in r.active]) for r in reqs]
    pool = kvq.PackedPool([r.T for r in dreqs], [r.active for r in dreqs], 8, 128, 4, dev)
    for j in range(4):
        kvq.kvq_encode_batch(pool, kvq.KVQ_K, j, kvq.pointer_array([r.xk[j] for r in dreqs], dev))
        kvq.kvq_encode_batch(pool, kvq.KVQ_V, j, kvq.pointer_array([r.xv[j] for r in dreqs], dev))
    outs = {k: [torch.empty((max(r.T, 1), 8, 128), dtype=torch.bfloat16, device=dev) for r in dreqs] for k in (0, 1)}
    for kind in (0, 1):
        kvq.kvq_reconstruct_batch(pool, kind, 4, kvq.pointer_array(outs[kind], dev))
    torch.cuda.synchronize()
    assert kvq.attn_error_word(pool.workspace) == 0
    for b, r in enumerate(dreqs):
        if r.T == 0:
            continue
        k1, v1 = P.gpu_chains(r)
        for j in range(4):
            for got, want in ((pool.k_streams[b][j], k1[j]), (pool.v_streams[b][j], v1[j])):
                assert torch.equal(got.codes_view(), want.codes_view())
                assert torch.equal(got.mins_view(), want.mins_view())
                assert torch.equal(got.scales_view(), want.scales_view())
                if want.sparse:
                    assert torch.equal(got.tile_dir_view(), want.tile_dir_view())
        assert torch.equal(outs[0][b][:r.T], kvq.kvq_reconstruct(k1, 4))
        assert torch.equal(outs[1][b][:r.T], kvq.kvq_reconstruct(v1, 4))
    q = W.make_queries(spec, 0, len(dreqs)).to(dev)
    live = [b for b in range(len(reqs)) if reqs[b].T > 0]
    ref = P.oracle_many([reqs[b] for b in live], q[live].cpu(), 4, P.softmax_scale(128), THREADS)
    for algo in _algos():
        out = kvq.kvq_decode_attn_packed(pool.table, q, 4, 8, algo=algo).cpu().numpy()
        assert np.all(out[[b for b in range(len(reqs)) if reqs[b].T == 0]] == 0)
        for j, b in enumerate(live):
            P.assert_attention_close(out[b], ref[j][4], f"pool req {b} algo {algo}")
