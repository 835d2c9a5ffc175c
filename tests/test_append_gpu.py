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
