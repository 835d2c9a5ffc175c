"""Codec edge values through the CUDA path vs the CPU oracle, bit for bit.

The sources exercise the corners of the quantiser and of the chain (FlashLoop
RFC, vllm-rlt issue #156, §3.3; INT4 codec PR, vllm-rlt pull #166): groups
whose min or max is a signed zero (the in-order scan keeps the first zero it
meets), constant groups of mixed-sign zeros, groups whose quotients are exact
half-integers (ties to even), a wide dynamic range inside a group, residuals
that vanish exactly, and chains deeper than four loops (kernels instantiated
for any depth)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_cross_loop_gb300 import kvq
from quantized_cross_loop_gb300.workloads import bf16_bits

from tests import pathrun as P

pytestmark = pytest.mark.gpu

D = 128


def special_source(T: int, H: int, seed: int) -> torch.Tensor:
    """BF16 [T, H, 128] whose heads hold one edge pattern each."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, D, generator=g)
    t = torch.arange(T).view(T, 1)
    c = torch.arange(D).view(1, D)
    sign = torch.where(torch.rand(T, D, generator=g) < 0.5, -1.0, 1.0)
    zeros = torch.zeros(T, D) * sign  # +0 and -0
    sprinkle = torch.rand(T, D, generator=g) < 0.1
    x[:, 0] = zeros  # constant groups of signed zeros
    x[:, 1] = torch.where(sprinkle, zeros, x[:, 1].abs())  # min is a signed zero
    x[:, 2] = torch.where(sprinkle, zeros, -x[:, 2].abs())  # max is a signed zero
    # every 64-row and every 64-channel group holds 0 and 15: scale 1, half-integer quotients
    x[:, 3] = ((t + c) % 31).float() / 2
    if H > 4:  # up to six decades inside one group
        x[:, 4] = x[:, 4] * torch.pow(10.0, torch.randint(-3, 4, (T, D), generator=g).float())
    if H > 5:  # ties again, negative and shifted
        x[:, 5] = -(((t + 3 * c) % 31).float() / 2) - 7.0
    return x.to(torch.bfloat16)


def nested(T: int, ratios, seed: int):
    g = torch.Generator().manual_seed(seed)
    sets, prev = [], None
    for r in ratios:
        if r >= 1.0:
            sets.append(None)
            continue
        pool = torch.arange(T) if prev is None else prev.to(torch.int64)
        n = min(pool.numel(), int(np.ceil(r * T)))
        cur = pool[torch.randperm(pool.numel(), generator=g)[:n]].sort().values.to(torch.int32)
        sets.append(cur)
        prev = cur
    return sets


def run_chain(kind, xs, actives):
    """GPU streams and oracle streams of one K or V chain."""
    gs = [kvq.kvq_encode_base(xs[0].cuda(), kind)]
    for r in range(1, len(xs)):
        act = actives[r]
        gs.append(kvq.kvq_encode_residual(xs[r].cuda(), gs, None if act is None else act.cuda()))
    os_ = O.encode_chain(kind, [bf16_bits(x) for x in xs],
                         [None if a is None else a.numpy().astype(np.int32) for a in actives])
    return gs, os_


def compare_chain(gs, os_, depths, what):
    for r in range(len(gs)):
        P.assert_stream_equal(gs[r], os_[r], f"{what} loop {r + 1}")
        P.assert_tile_dir(gs[r])
    for depth in depths:
        got = bf16_bits(kvq.kvq_reconstruct(gs, depth))
        assert np.array_equal(got, O.reconstruct(os_, depth)), f"{what} reconstruct depth {depth}"


@pytest.mark.parametrize("T", [64, 200])
@pytest.mark.parametrize("kind", [kvq.KVQ_K, kvq.KVQ_V])
def test_special_values_chain(T, kind):
    H = 8
    xs = [special_source(T, H, 11 + T)]
    g = torch.Generator().manual_seed(100 + T)
    for _ in range(1, 4):
        xs.append((xs[-1].float() + 0.1 * torch.randn(xs[-1].shape, generator=g)).to(torch.bfloat16))
    # loop 2 equals the reconstruction of loop 1 on heads 0 and 1 (exactly vanishing residuals,
    # some of them perturbed), so the residual groups are constant +0 or have a zero min/max
    s1 = O.encode(kind, bf16_bits(xs[0]))
    xhat1 = torch.from_numpy(O.reconstruct([s1], 1).astype(np.int16)).view(torch.bfloat16)
    x2 = xs[1].clone()
    x2[:, 0] = xhat1[:, 0]
    bump = torch.rand(T, D, generator=g) < 0.05
    x2[:, 1] = torch.where(bump, (xhat1[:, 1].float() + 0.25).to(torch.bfloat16), xhat1[:, 1])
    xs[1] = x2
    actives = nested(T, (1.0, 1.0, 0.5, 0.25), 7 + T)
    gs, os_ = run_chain(kind, xs, actives)
    compare_chain(gs, os_, (1, 2, 3, 4), f"kind {kind} T {T}")


@pytest.mark.parametrize("kind", [kvq.KVQ_K, kvq.KVQ_V])
def test_deep_chain(kind):
    """Six loops: loops 5-6 and depths 5-6 run the any-depth kernels; depth 4 the fast ones."""
    T, H = 150, 4
    g = torch.Generator().manual_seed(5)
    x = torch.randn(T, H, D, generator=g)
    xs = [x.to(torch.bfloat16)]
    for _ in range(1, 6):
        x = x + 0.1 * torch.randn(T, H, D, generator=g)
        xs.append(x.to(torch.bfloat16))
    actives = nested(T, (1.0, 1.0, 0.5, 0.25, 0.1, 0.05), 9)
    gs, os_ = run_chain(kind, xs, actives)
    compare_chain(gs, os_, (4, 5, 6), f"deep kind {kind}")


def test_batch_deep_chain_matches_single():
    """Batched encode and reconstruction of five loops (the fifth through the
    any-depth kernels) give the bytes of the per-request calls."""
    H, loops = 8, 5
    dev = torch.device("cuda")
    lengths = [130, 1, 64, 300]
    xs_all, act_all = [], []
    for b, T in enumerate(lengths):
        g = torch.Generator().manual_seed(21 + b)
        per = {}
        for kind in (kvq.KVQ_K, kvq.KVQ_V):
            x = torch.randn(T, H, D, generator=g)
            seq = [x.to(torch.bfloat16)]
            for _ in range(1, loops):
                x = x + 0.1 * torch.randn(T, H, D, generator=g)
                seq.append(x.to(torch.bfloat16))
            per[kind] = [t.to(dev) for t in seq]
        xs_all.append(per)
        act_all.append([None if a is None else a.to(dev) for a in nested(T, (1.0, 1.0, 0.5, 0.25, 0.2), 3 + b)])
    pool = kvq.PackedPool(lengths, act_all, H, D, loops, dev)
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
            gs = [kvq.kvq_encode_base(xs[0], kind)]
            for r in range(1, loops):
                gs.append(kvq.kvq_encode_residual(xs[r], gs, act_all[b][r]))
            for j in range(loops):
                assert torch.equal(pstreams[j].codes_view(), gs[j].codes_view()), f"req {b} kind {kind} loop {j}"
                assert torch.equal(pstreams[j].mins_view(), gs[j].mins_view())
                assert torch.equal(pstreams[j].scales_view(), gs[j].scales_view())
            assert torch.equal(outs[kind][b], kvq.kvq_reconstruct(gs, loops)), f"req {b} kind {kind}"
