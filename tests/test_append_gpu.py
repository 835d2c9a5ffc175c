"""Appending 64-token tiles to packed chains in place (FlashLoop RFC, vllm-rlt
issue #156, §3.3: the rolling BF16 tail is flushed into the packed form in
whole 64-token groups), through the C ABI: after the appends every plane holds
the bytes of the oracle's encode of the whole extended chain (tile-local K
grouping, INT4 codec PR review), the reconstruction is bit-exact and the
attention over the grown chain matches the oracle."""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_cross_loop_gb300 import kvq
from quantized_cross_loop_gb300.workloads import bf16_bits

from tests import pathrun as P
from tests.test_codec_edge_gpu import nested
from tests.test_kgroup_tile_gpu import drift

pytestmark = pytest.mark.gpu

D = 128
TILE = kvq.KVQ_KGROUP_TILE


def grow_chain(kind, xs, actives, T0, n_tiles, kgroup=TILE):
    """Encode the first T0 tokens with room for n_tiles more, then append them tile by tile."""
    Ttot = T0 + 64 * n_tiles
    dev = torch.device("cuda")
    gs = [kvq.kvq_encode_base(xs[0][:T0].cuda(), kind, kgroup=kgroup, token_cap=Ttot)]
    for r in range(1, len(xs)):
        a = actives[r]
        a0 = None if a is None else a[a < T0].contiguous()
        gs.append(kvq.kvq_encode_residual(xs[r][:T0].cuda(), gs, None if a0 is None else a0.cuda(),
                                          row_cap=Ttot, token_cap=Ttot))
    for k in range(n_tiles):
        t0 = T0 + 64 * k
        x_tile = [x[t0:t0 + 64].contiguous().to(dev) for x in xs]
        rel = [None if a is None else (a[(a >= t0) & (a < t0 + 64)] - t0).to(torch.int32) for a in actives]
        ws = kvq.kvq_append_tile(gs, x_tile, rel)
        torch.cuda.synchronize()
        assert kvq.attn_error_word(ws) == 0
    return gs


def oracle_chain(kind, xs, actives):
    return O.encode_chain(kind, [bf16_bits(x) for x in xs],
                          [None if a is None else a.numpy().astype(np.int32) for a in actives], kgroup=O.KGROUP_TILE)


@pytest.mark.parametrize("T0,n_tiles,ratios", [
    (256, 3, (1.0, 1.0, 0.5, 0.25)),
    (0, 4, (1.0, 1.0, 0.5, 0.25)),      # the packed chain starts empty
    (128, 2, (1.0, 1.0, 0.1, 0.02)),    # sparse loops with tiles that store no row
    (64, 1, (1.0, 1.0, 1.0, 1.0)),
])
@pytest.mark.parametrize("kind", [kvq.KVQ_K, kvq.KVQ_V])
def test_append_tiles_equal_full_encode(T0, n_tiles, ratios, kind):
    H = 8
    Ttot = T0 + 64 * n_tiles
    xs = drift(Ttot, H, 4, 900 + T0 + kind)
    actives = nested(Ttot, ratios, 901 + T0)
    gs = grow_chain(kind, xs, actives, T0, n_tiles)
    os_ = oracle_chain(kind, xs, actives)
    for r in range(4):
        assert gs[r].n_tokens == Ttot and gs[r].n_rows == os_[r].n
        P.assert_stream_equal(gs[r], os_[r], f"T0 {T0} kind {kind} loop {r + 1}")
        P.assert_tile_dir(gs[r])
    for depth in (1, 2, 4):
        got = bf16_bits(kvq.kvq_reconstruct(gs, depth))
        assert np.array_equal(got, O.reconstruct(os_, depth)), f"reconstruct depth {depth}"


def test_attention_over_grown_chains():
    """Two requests grown by appends, read by both attention kernels at depth 4."""
    H, Hq = 8, 32
    kc, vc, oks, ovs = [], [], [], []
    for b, (T0, n) in enumerate([(320, 2), (0, 3)]):
        Ttot = T0 + 64 * n
        actives = nested(Ttot, (1.0, 1.0, 0.5, 0.25), 950 + b)
        for kind, chains, orc in ((kvq.KVQ_K, kc, oks), (kvq.KVQ_V, vc, ovs)):
            xs = drift(Ttot, H, 4, 960 + 2 * b + kind)
            chains.append(grow_chain(kind, xs, actives, T0, n))
            orc.append(oracle_chain(kind, xs, actives))
    table = kvq.RequestTable(kc, vc, torch.device("cuda"))
    q = torch.randn((2, Hq, D), generator=torch.Generator().manual_seed(970)).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    for algo in (kvq.ATTN_SIMT, kvq.ATTN_MMA):
        ws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(2, H, Hq, D), dtype=torch.uint8, device="cuda")
        out = kvq.kvq_decode_attn_packed(table, q.cuda(), 4, H, algo=algo, workspace=ws).cpu().numpy()
        assert kvq.attn_error_word(ws) == 0
        for b in range(2):
            ref = O.attention_f32(bf16_bits(q[b]), O.decode_f32(oks[b], 4), O.decode_f32(ovs[b], 4), scale)
            P.assert_attention_close(out[b], ref, f"req {b} algo {algo}")


def test_append_refusals():
    """Host checks: compact-grouped sparse K, a length that is not a multiple of 64,
    too little capacity and NVFP4 loops are refused before any launch."""
    H, T0 = 8, 128
    xs = drift(T0 + 64, H, 3, 990)
    act = nested(T0 + 64, (1.0, 1.0, 0.5), 991)
    dev = torch.device("cuda")
    x_tile = [x[T0:].contiguous().to(dev) for x in xs]
    rel = [None, None, (act[2][act[2] >= T0] - T0).to(torch.int32)]

    def chain(kgroup, fmt=kvq.KVQ_FMT_INT4, cap=T0 + 64, T=T0):
        gs = [kvq.kvq_encode_base(xs[0][:T].cuda(), kvq.KVQ_K, kgroup=kgroup, token_cap=cap)]
        gs.append(kvq.kvq_encode_residual(xs[1][:T].cuda(), gs, row_cap=cap, token_cap=cap, fmt=fmt))
        a = act[2][act[2] < T].contiguous().cuda()
        gs.append(kvq.kvq_encode_residual(xs[2][:T].cuda(), gs, a, row_cap=cap, token_cap=cap))
        return gs

    with pytest.raises(kvq.KvqError, match="tile grouping"):
        kvq.kvq_append_tile(chain(kvq.KVQ_KGROUP_COMPACT), x_tile, rel)
    with pytest.raises(kvq.KvqError, match="capacities"):
        kvq.kvq_append_tile(chain(TILE, cap=T0 + 32), x_tile, rel)
    with pytest.raises(kvq.KvqError, match="NVFP4"):
        kvq.kvq_append_tile(chain(TILE, fmt=kvq.KVQ_FMT_NVFP4), x_tile, rel)
    with pytest.raises(kvq.KvqError, match="multiple"):
        kvq.kvq_append_tile(chain(TILE, T=T0 - 8, cap=T0 + 64), x_tile, rel)


def test_batched_append_equals_full_encode():
    """kvq_append_tile_batch: tiles appended to every request of a pool in one call
    per tile give the bytes of the oracle's encode of each whole chain (K and V),
    update the device table, and the attention reads the grown chains."""
    H, D_, loops = 8, 128, 4
    dev = torch.device("cuda")
    lengths0 = [256, 0, 128, 320, 64]
    n_tiles = 2
    caps = [T + 64 * n_tiles for T in lengths0]
    xs_all, act_all = [], []
    for b, Ttot in enumerate(caps):
        xs_all.append({kind: drift(Ttot, H, loops, 1100 + 2 * b + kind) for kind in (0, 1)})
        act_all.append(nested(Ttot, (1.0, 1.0, 0.5, 0.1), 1110 + b))
    act0 = [[None if a is None else a[a < lengths0[b]].contiguous().to(dev) for a in act_all[b]]
            for b in range(len(caps))]
    pool = kvq.PackedPool(lengths0, act0, H, D_, loops, dev, kgroup=TILE, token_caps=caps)
    for j in range(loops):
        for kind in (kvq.KVQ_K, kvq.KVQ_V):
            kvq.kvq_encode_batch(pool, kind, j, kvq.pointer_array(
                [xs_all[b][kind][j][:lengths0[b]].contiguous().to(dev) for b in range(len(caps))], dev))
    for k in range(n_tiles):
        xk = [[None] * len(caps) for _ in range(loops)]
        xv = [[None] * len(caps) for _ in range(loops)]
        rel = [[None] * len(caps) for _ in range(loops)]
        for b in range(len(caps)):
            t0 = lengths0[b] + 64 * k
            for j in range(loops):
                xk[j][b] = xs_all[b][0][j][t0:t0 + 64].contiguous().to(dev)
                xv[j][b] = xs_all[b][1][j][t0:t0 + 64].contiguous().to(dev)
                a = act_all[b][j]
                rel[j][b] = None if a is None else (a[(a >= t0) & (a < t0 + 64)] - t0).to(torch.int32)
        ws = pool.append_tile(xk, xv, rel)
        torch.cuda.synchronize()
        assert kvq.attn_error_word(ws) == 0
    pool.sync_counts()
    for b, Ttot in enumerate(caps):
        assert pool.lengths[b] == Ttot
        for kind, streams in ((kvq.KVQ_K, pool.k_streams[b]), (kvq.KVQ_V, pool.v_streams[b])):
            os_ = oracle_chain(kind, xs_all[b][kind], act_all[b])
            for r in range(loops):
                P.assert_stream_equal(streams[r], os_[r], f"req {b} kind {kind} loop {r + 1}")
                P.assert_tile_dir(streams[r])
    # the device table already describes the grown chains
    Hq = 32
    q = torch.randn((len(caps), Hq, D_), generator=torch.Generator().manual_seed(1120)).to(torch.bfloat16)
    out = kvq.kvq_decode_attn_packed(pool.table, q.cuda(), 4, H, algo=kvq.ATTN_MMA).cpu().numpy()
    scale = 1.0 / math.sqrt(D_)
    for b in range(len(caps)):
        ok_ = oracle_chain(kvq.KVQ_K, xs_all[b][0], act_all[b])
        ov_ = oracle_chain(kvq.KVQ_V, xs_all[b][1], act_all[b])
        ref = O.attention_f32(bf16_bits(q[b]), O.decode_f32(ok_, 4), O.decode_f32(ov_, 4), scale)
        P.assert_attention_close(out[b], ref, f"req {b}")


def test_batched_append_refuses_per_request():
    """A request without room for the tile is left unchanged (error bit 1); the
    others grow."""
    H, D_, loops = 8, 128, 2
    dev = torch.device("cuda")
    lengths0 = [128, 64]
    caps = [192, 64]  # request 1 has no room
    xs = [drift(c if c > L else L + 64, H, loops, 1200 + b) for b, (L, c) in enumerate(zip(lengths0, caps))]
    pool = kvq.PackedPool(lengths0, [[None, None]] * 2, H, D_, loops, dev, kgroup=TILE, token_caps=caps)
    for j in range(loops):
        ptr = kvq.pointer_array([xs[b][j][:lengths0[b]].contiguous().to(dev) for b in range(2)], dev)
        kvq.kvq_encode_batch(pool, kvq.KVQ_K, j, ptr)
        kvq.kvq_encode_batch(pool, kvq.KVQ_V, j, ptr)
    tiles = [[xs[b][j][lengths0[b]:lengths0[b] + 64].contiguous().to(dev) for b in range(2)] for j in range(loops)]
    ws = pool.append_tile(tiles, tiles, [[None, None]] * loops)
    torch.cuda.synchronize()
    assert kvq.attn_error_word(ws) & 1
    pool.sync_counts()
    assert pool.lengths == [192, 64]
