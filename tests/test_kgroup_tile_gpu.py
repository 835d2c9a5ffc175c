"""Tile-local K grouping (INT4 codec PR, vllm-rlt pull #166, review by 0z5a:
group ownership vs 16-token pages) through the C ABI against the oracle: a
sparse K residual's groups hold the stored rows of one 64-token logical tile,
so a tile's rows and metadata never depend on another tile.

Codec planes and reconstructions must be bit-exact; attention (both kernels)
and sparse decode attention within |gpu - oracle| <= 2e-3 + 1e-2 * |oracle|."""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_cross_loop_gb300 import kvq
from quantized_cross_loop_gb300.workloads import bf16_bits

from tests import pathrun as P
from tests.test_codec_edge_gpu import nested, special_source

pytestmark = pytest.mark.gpu

D = 128
TILE = kvq.KVQ_KGROUP_TILE


def drift(T, H, loops, seed, sigma=0.1):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, D, generator=g)
    xs = [x.to(torch.bfloat16)]
    for _ in range(1, loops):
        x = x + sigma * torch.randn(T, H, D, generator=g)
        xs.append(x.to(torch.bfloat16))
    return xs


def drop_tiles(act, tiles):
    """Remove every index of the given 64-token tiles from an active set."""
    if act is None:
        return None
    keep = torch.ones(act.numel(), dtype=torch.bool)
    for k in tiles:
        keep &= (act // 64) != k
    return act[keep].contiguous()


def run_tile_chain(kind, xs, actives):
    gs = [kvq.kvq_encode_base(xs[0].cuda(), kind, kgroup=TILE)]
    for r in range(1, len(xs)):
        act = actives[r]
        gs.append(kvq.kvq_encode_residual(xs[r].cuda(), gs, None if act is None else act.cuda()))
    os_ = O.encode_chain(kind, [bf16_bits(x) for x in xs],
                         [None if a is None else a.numpy().astype(np.int32) for a in actives], kgroup=O.KGROUP_TILE)
    return gs, os_


def compare(gs, os_, depths, what):
    for r in range(len(gs)):
        P.assert_stream_equal(gs[r], os_[r], f"{what} loop {r + 1}")
        P.assert_tile_dir(gs[r])
    for depth in depths:
        got = bf16_bits(kvq.kvq_reconstruct(gs, depth))
        assert np.array_equal(got, O.reconstruct(os_, depth)), f"{what} reconstruct depth {depth}"


@pytest.mark.parametrize("T,ratios,dropped", [
    (1000, (1.0, 1.0, 0.5, 0.25), ()),        # partial last tile, nested random sets
    (300, (1.0, 1.0, 0.5, 0.25), (2,)),       # a tile with no stored row in loops 3 and 4
    (65, (1.0, 1.0, 0.5, 0.1), ()),           # one token in the last tile
    (1, (1.0, 1.0, 1.0, 1.0), ()),
    (4096, (1.0, 1.0, 0.05, 0.01), (5, 6, 7)),  # very sparse: most tiles hold 0-5 rows
])
def test_tile_grouped_chain_bit_exact(T, ratios, dropped):
    H = 8
    actives = [drop_tiles(a, dropped) for a in nested(T, ratios, 31 + T)]
    for kind, xs in ((kvq.KVQ_K, drift(T, H, 4, 40 + T)), (kvq.KVQ_V, drift(T, H, 4, 50 + T))):
        gs, os_ = run_tile_chain(kind, xs, actives)
        compare(gs, os_, (1, 2, 3, 4), f"T {T} kind {kind}")


def test_tile_grouped_special_values():
    """Exact ties, signed zeros and wide ranges inside the tile groups."""
    T, H = 200, 8
    xs = [special_source(T, H, 77)]
    g = torch.Generator().manual_seed(78)
    for _ in range(1, 4):
        xs.append((xs[-1].float() + 0.1 * torch.randn(xs[-1].shape, generator=g)).to(torch.bfloat16))
    actives = nested(T, (1.0, 1.0, 0.5, 0.25), 79)
    gs, os_ = run_tile_chain(kvq.KVQ_K, xs, actives)
    compare(gs, os_, (2, 3, 4), "special")


def test_tile_grouped_deep_chain():
    """Six loops: loops 5-6 and depths 5-6 through the any-depth kernels."""
    T, H = 150, 4
    actives = nested(T, (1.0, 1.0, 0.5, 0.25, 0.1, 0.05), 81)
    gs, os_ = run_tile_chain(kvq.KVQ_K, drift(T, H, 6, 82), actives)
    compare(gs, os_, (4, 5, 6), "deep")


def test_tile_grouped_batch_matches_single():
    """Batched encode and reconstruction under tile grouping give the bytes of
    the per-request calls; one request has an empty loop-4 set."""
    H, loops = 8, 4
    dev = torch.device("cuda")
    lengths = [1000, 130, 64, 300]
    xs_all, act_all = [], []
    for b, T in enumerate(lengths):
        xs_all.append({kind: [t.to(dev) for t in drift(T, H, loops, 90 + 2 * b + kind)] for kind in (0, 1)})
        acts = nested(T, (1.0, 1.0, 0.5, 0.25), 95 + b)
        if b == 2:
            acts[3] = torch.zeros(0, dtype=torch.int32)
        act_all.append([None if a is None else a.to(dev) for a in acts])
    pool = kvq.PackedPool(lengths, act_all, H, D, loops, dev, kgroup=TILE)
    for j in range(loops):
        for kind in (kvq.KVQ_K, kvq.KVQ_V):
            kvq.kvq_encode_batch(pool, kind, j, kvq.pointer_array([xs_all[b][kind][j] for b in range(len(lengths))], dev))
    outs = {k: [torch.empty((T, H, D), dtype=torch.bfloat16, device=dev) for T in lengths] for k in (0, 1)}
    for kind in (kvq.KVQ_K, kvq.KVQ_V):
        kvq.kvq_reconstruct_batch(pool, kind, loops, kvq.pointer_array(outs[kind], dev))
    torch.cuda.synchronize()
    assert kvq.attn_error_word(pool.workspace) == 0
    for b in range(len(lengths)):
        for kind, pstreams in ((kvq.KVQ_K, pool.k_streams[b]), (kvq.KVQ_V, pool.v_streams[b])):
            xs = xs_all[b][kind]
            gs = [kvq.kvq_encode_base(xs[0], kind, kgroup=TILE)]
            for r in range(1, loops):
                gs.append(kvq.kvq_encode_residual(xs[r], gs, act_all[b][r]))
            for j in range(loops):
                assert torch.equal(pstreams[j].codes_view(), gs[j].codes_view()), f"req {b} kind {kind} loop {j}"
                assert torch.equal(pstreams[j].mins_view(), gs[j].mins_view())
                assert torch.equal(pstreams[j].scales_view(), gs[j].scales_view())
            assert torch.equal(outs[kind][b], kvq.kvq_reconstruct(gs, loops)), f"req {b} kind {kind}"


def _tile_requests(lengths, Hq, seed):
    H = 8
    kc, vc, oks, ovs = [], [], [], []
    for b, T in enumerate(lengths):
        actives = [drop_tiles(a, (1,)) for a in nested(T, (1.0, 1.0, 0.5, 0.25), seed + b)]
        for kind, chains, orc in ((kvq.KVQ_K, kc, oks), (kvq.KVQ_V, vc, ovs)):
            gs, os_ = run_tile_chain(kind, drift(T, H, 4, seed + 10 * b + kind), actives)
            chains.append(gs)
            orc.append(os_)
    q = torch.randn((len(lengths), Hq, D), generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    return H, kc, vc, oks, ovs, q


@pytest.mark.parametrize("Hq", [32, 64])
def test_tile_grouped_attention(Hq):
    """Both attention kernels read tile-grouped K params (the tensor-core
    kernel stages one K group per tile and loop) at every depth."""
    lengths = [1000, 4096, 130, 1]
    H, kc, vc, oks, ovs, q = _tile_requests(lengths, Hq, 300 + Hq)
    table = kvq.RequestTable(kc, vc, torch.device("cuda"))
    scale = 1.0 / math.sqrt(D)
    for depth in (2, 3, 4):
        for algo in (kvq.ATTN_SIMT, kvq.ATTN_MMA):
            ws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(len(lengths), H, Hq, D), dtype=torch.uint8,
                             device="cuda")
            out = kvq.kvq_decode_attn_packed(table, q.cuda(), depth, H, algo=algo, workspace=ws)
            torch.cuda.synchronize()
            assert kvq.attn_error_word(ws) == 0
            out = out.cpu().numpy()
            for b in range(len(lengths)):
                ref = O.attention_f32(bf16_bits(q[b]), O.decode_f32(oks[b], depth), O.decode_f32(ovs[b], depth),
                                      scale)
                P.assert_attention_close(out[b], ref, f"req {b} depth {depth} algo {algo}")


def test_tile_grouped_sparse_decode():
    """Sparse decode attention (FlashLoop RFC §3.2) on tile-grouped chains: the
    later loop's output from the GPU state matches the oracle's correction."""
    lengths = [1000, 300]
    Hq = 32
    H, kc, vc, oks, ovs, q = _tile_requests(lengths, Hq, 500)
    table = kvq.RequestTable(kc, vc, torch.device("cuda"))
    scale = 1.0 / math.sqrt(D)
    st = kvq.kvq_sparse_ref_state(table, q.cuda(), 2, H, 128, max(lengths))
    q4 = torch.randn((len(lengths), Hq, D), generator=torch.Generator().manual_seed(501)).to(torch.bfloat16)
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")  # the per-key kernel
    out = kvq.kvq_sparse_decode_attn(table, q4.cuda(), 4, H, st, workspace=ws).cpu().numpy()
    wsb = torch.zeros(kvq.kvq_sparse_decode_workspace_bytes(len(lengths), H, Hq, D, max(lengths)), dtype=torch.uint8,
                      device="cuda")  # the key-masked tensor-core attention
    out_tc = kvq.kvq_sparse_decode_attn(table, q4.cuda(), 4, H, st, workspace=wsb, algo=kvq.ATTN_MMA).cpu().numpy()
    torch.cuda.synchronize()
    assert kvq.attn_error_word(st.workspace) == 0 and kvq.attn_error_word(ws) == 0 and kvq.attn_error_word(wsb) == 0
    sel, mass, o_ref, c_ref = (t.cpu().numpy() for t in (st.sel_idx, st.mass, st.o_ref, st.c_ref))
    for b, T in enumerate(lengths):
        K = min(128, T)
        S = sel[b][:, :K]
        kf2, vf2 = O.decode_f32(oks[b], 2), O.decode_f32(ovs[b], 2)
        # O_ref against the oracle attention at the reference depth
        P.assert_attention_close(o_ref[b], O.attention_f32(bf16_bits(q[b]), kf2, vf2, scale), f"O_ref req {b}")
        ref = O.sparse_decode(bf16_bits(q4[b]), O.decode_f32(oks[b], 4), O.decode_f32(ovs[b], 4), scale, S,
                              mass[b].astype(np.float64), o_ref[b].astype(np.float64), c_ref[b].astype(np.float64))
        P.assert_attention_close(out[b], ref, f"sparse req {b}")
        P.assert_attention_close(out_tc[b], ref, f"sparse req {b}, tensor-core path")
