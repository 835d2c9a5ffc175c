"""NVFP4 residual loops (INT4 codec PR, vllm-rlt pull #166, review by 0z5a:
E2M1 elements, one E4M3 scale per 16 channels, one FP32 scale per stream;
INT4 base plus NVFP4 residuals) through the C ABI against the oracle.

Codes, E4M3 block scales, the tensor scale and the BF16 reconstructions must be
bit-exact; attention within |gpu - oracle| <= 2e-3 + 1e-2 * |oracle| of the
oracle's FP32 decode of the same packed chain."""

from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_cross_loop_gb300 import kvq
from quantized_cross_loop_gb300.workloads import bf16_bits

from tests import pathrun as P
from tests.test_codec_edge_gpu import nested, special_source
from tests.test_kgroup_tile_gpu import drift

pytestmark = pytest.mark.gpu

D = 128
NV, I4 = kvq.KVQ_FMT_NVFP4, kvq.KVQ_FMT_INT4


def run_chain(kind, xs, actives, formats, kgroup=kvq.KVQ_KGROUP_COMPACT):
    gs = [kvq.kvq_encode_base(xs[0].cuda(), kind, kgroup=kgroup)]
    for r in range(1, len(xs)):
        act = actives[r]
        gs.append(kvq.kvq_encode_residual(xs[r].cuda(), gs, None if act is None else act.cuda(), fmt=formats[r]))
    os_ = O.encode_chain(kind, [bf16_bits(x) for x in xs],
                         [None if a is None else a.numpy().astype(np.int32) for a in actives],
                         kgroup=O.KGROUP_TILE if kgroup == kvq.KVQ_KGROUP_TILE else O.KGROUP_COMPACT,
                         formats=[O.FMT_NVFP4 if f == NV else O.FMT_INT4 for f in formats])
    return gs, os_


def assert_stream(gs, os_, what):
    if os_.fmt != O.FMT_NVFP4:
        P.assert_stream_equal(gs, os_, what)
        return
    assert np.array_equal(gs.codes_view().cpu().numpy(), os_.codes), f"codes differ {what}"
    assert np.array_equal(gs.mins_view().cpu().numpy(), os_.bscale), f"block scales differ {what}"
    assert gs.scales_view().cpu().numpy()[0].view(np.uint32) == os_.tscale[0].view(np.uint32), f"s_t differs {what}"


def compare(gs, os_, depths, what):
    for r in range(len(gs)):
        assert_stream(gs[r], os_[r], f"{what} loop {r + 1}")
        P.assert_tile_dir(gs[r])
    for depth in depths:
        got = bf16_bits(kvq.kvq_reconstruct(gs, depth))
        assert np.array_equal(got, O.reconstruct(os_, depth)), f"{what} reconstruct depth {depth}"


@pytest.mark.parametrize("T,ratios,formats", [
    (1000, (1.0, 1.0, 0.5, 0.25), (I4, NV, NV, NV)),  # INT4 base + NVFP4 residuals, sparse late loops
    (1000, (1.0, 1.0, 0.5, 0.25), (I4, I4, NV, I4)),  # mixed: an INT4 loop after an NVFP4 one
    (65, (1.0, 1.0, 0.5, 0.1), (I4, NV, NV, NV)),
    (1, (1.0, 1.0, 1.0, 1.0), (I4, NV, NV, NV)),
])
@pytest.mark.parametrize("kind", [kvq.KVQ_K, kvq.KVQ_V])
def test_nvfp4_chain_bit_exact(T, ratios, formats, kind):
    H = 8
    actives = nested(T, ratios, 61 + T)
    gs, os_ = run_chain(kind, drift(T, H, 4, 70 + T + kind), actives, formats)
    compare(gs, os_, (2, 3, 4), f"T {T} kind {kind} formats {formats}")


def test_nvfp4_special_values():
    """Exactly vanishing residuals (a zero tensor scale on some heads' blocks and
    E2M1 ties), signed zeros and six decades of range inside a stream."""
    T, H = 200, 8
    xs = [special_source(T, H, 88)]
    g = torch.Generator().manual_seed(89)
    for _ in range(1, 4):
        xs.append((xs[-1].float() + 0.1 * torch.randn(xs[-1].shape, generator=g)).to(torch.bfloat16))
    s1 = O.encode(O.KIND_V, bf16_bits(xs[0]))
    xhat1 = torch.from_numpy(O.reconstruct([s1], 1).astype(np.int16)).view(torch.bfloat16)
    x2 = xs[1].clone()
    x2[:, 0] = xhat1[:, 0]  # head 0: residual exactly zero
    xs[1] = x2
    actives = nested(T, (1.0, 1.0, 0.5, 0.25), 90)
    for kind in (kvq.KVQ_K, kvq.KVQ_V):
        gs, os_ = run_chain(kind, xs, actives, (I4, NV, NV, NV))
        compare(gs, os_, (2, 4), f"special kind {kind}")
    # a residual that vanishes everywhere: tensor scale 0, every code and scale 0
    gs = [kvq.kvq_encode_base(xs[0].cuda(), kvq.KVQ_V)]
    z = kvq.kvq_encode_residual(kvq.kvq_reconstruct(gs, 1), gs, fmt=NV)
    torch.cuda.synchronize()
    assert float(z.scales_view()[0]) == 0.0 and not z.codes_view().any() and not z.mins_view().any()


def test_nvfp4_deep_and_tile_grouped():
    """Six loops (any-depth kernels) with NVFP4 residuals over a tile-grouped INT4 base."""
    T, H = 150, 4
    actives = nested(T, (1.0, 1.0, 0.5, 0.25, 0.1, 0.05), 91)
    formats = (I4, NV, I4, NV, NV, I4)
    gs, os_ = run_chain(kvq.KVQ_K, drift(T, H, 6, 92), actives, formats, kgroup=kvq.KVQ_KGROUP_TILE)
    compare(gs, os_, (4, 5, 6), "deep")


def test_nvfp4_batch_matches_single():
    """Batched encode and reconstruction of INT4-base + NVFP4-residual chains give
    the bytes of the per-request calls; the INT4-only entry point refuses them."""
    H, loops = 8, 4
    dev = torch.device("cuda")
    lengths = [1000, 130, 64, 300]
    formats = [I4, NV, NV, NV]
    xs_all, act_all = [], []
    for b, T in enumerate(lengths):
        xs_all.append({kind: [t.to(dev) for t in drift(T, H, loops, 110 + 2 * b + kind)] for kind in (0, 1)})
        act_all.append([None if a is None else a.to(dev) for a in nested(T, (1.0, 1.0, 0.5, 0.25), 115 + b)])
    pool = kvq.PackedPool(lengths, act_all, H, D, loops, dev, formats=formats)
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
                gs.append(kvq.kvq_encode_residual(xs[r], gs, act_all[b][r], fmt=formats[r]))
            for j in range(loops):
                assert torch.equal(pstreams[j].codes_view(), gs[j].codes_view()), f"req {b} kind {kind} loop {j}"
                assert torch.equal(pstreams[j].mins_view(), gs[j].mins_view())
                assert torch.equal(pstreams[j].scales_view(), gs[j].scales_view())
            assert torch.equal(outs[kind][b], kvq.kvq_reconstruct(gs, loops)), f"req {b} kind {kind}"
    # the INT4-only batch entry refuses the NVFP4 loops: error bit 64, nothing written
    ws = torch.zeros_like(pool.workspace)
    L = kvq.lib()
    st = L.kvq_reconstruct_batch(kvq._dptr(pool.table.table), pool.n_requests, H, D, kvq.KVQ_K, loops,
                                 kvq._dptr(kvq.pointer_array(outs[0], dev)), kvq._dptr(ws), ws.numel(), None)
    torch.cuda.synchronize()
    assert st == 0 and kvq.attn_error_word(ws) & 64


def _nvfp4_requests(lengths, Hq, seed, formats=(I4, NV, NV, NV)):
    H = 8
    kc, vc, oks, ovs = [], [], [], []
    for b, T in enumerate(lengths):
        actives = nested(T, (1.0, 1.0, 0.5, 0.25), seed + b)
        for kind, chains, orc in ((kvq.KVQ_K, kc, oks), (kvq.KVQ_V, vc, ovs)):
            gs, os_ = run_chain(kind, drift(T, H, 4, seed + 10 * b + kind), actives, formats)
            chains.append(gs)
            orc.append(os_)
    q = torch.randn((len(lengths), Hq, D), generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    return H, kc, vc, oks, ovs, q


@pytest.mark.parametrize("Hq", [32, 64])
@pytest.mark.parametrize("formats", [(I4, NV, NV, NV), (I4, I4, NV, I4)])
def test_nvfp4_attention(Hq, formats):
    """Both attention kernels read NVFP4 loops (the tensor-core kernel in its
    NVFP4 form, scaling the A operands by the E4M3 block scales) at every depth."""
    lengths = [1000, 4096, 130, 1]
    H, kc, vc, oks, ovs, q = _nvfp4_requests(lengths, Hq, 400 + Hq, formats)
    table = kvq.RequestTable(kc, vc, torch.device("cuda"))
    assert table.has_nvfp4
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


def test_int4_tensor_core_kernel_refuses_nvfp4():
    """Without the NVFP4 hint the INT4 tensor-core kernel reads no NVFP4 plane: the
    request's output is NaN and error bit 64 is set; the INT4 request beside it is exact."""
    H, Hq = 8, 32
    _, kc, vc, oks, ovs, q = _nvfp4_requests([300], Hq, 700)
    _, kc4, vc4, oks4, ovs4, _ = _nvfp4_requests([200], Hq, 701, (I4, I4, I4, I4))
    table = kvq.RequestTable(kc + kc4, vc + vc4, torch.device("cuda"))
    q2 = torch.randn((2, Hq, D), generator=torch.Generator().manual_seed(702)).to(torch.bfloat16).cuda()
    ws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(2, H, Hq, D), dtype=torch.uint8, device="cuda")
    out = torch.empty((2, Hq, D), dtype=torch.float32, device="cuda")
    L = kvq.lib()
    st = L.kvq_decode_attn_packed_ex(kvq._dptr(table.table), 2, H, Hq, D, 4, kvq._dptr(q2), ctypes.c_float(0.088),
                                     kvq._dptr(out), kvq._dptr(ws), ws.numel(), kvq.ATTN_MMA, None)
    torch.cuda.synchronize()
    assert st == 0 and kvq.attn_error_word(ws) & 64
    o = out.cpu().numpy()
    assert np.all(np.isnan(o[0]))
    ref = O.attention_f32(bf16_bits(q2[1].cpu()), O.decode_f32(oks4[0], 4), O.decode_f32(ovs4[0], 4), 0.088)
    P.assert_attention_close(o[1], ref, "INT4 request")


def test_nvfp4_flag_picks_the_kernel_on_the_device():
    """With KVQ_ATTN_NVFP4 the call launches the INT4 kernel and the NVFP4-reading
    one, and the plan picks the one that works: an INT4 table gives the bits of
    the call without the flag, a table holding an NVFP4 loop those of the general
    kernel (which reads both formats); either within the attention tolerance of
    the oracle."""
    H, Hq = 8, 32
    _, kc, vc, oks, ovs, _ = _nvfp4_requests([300], Hq, 720)
    _, kc4, vc4, oks4, ovs4, _ = _nvfp4_requests([200, 77], Hq, 721, (I4, I4, I4, I4))
    q3 = torch.randn((3, Hq, D), generator=torch.Generator().manual_seed(722)).to(torch.bfloat16).cuda()
    L = kvq.lib()

    def call(table, n, algo):
        ws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(n, H, Hq, D), dtype=torch.uint8, device="cuda")
        out = torch.empty((n, Hq, D), dtype=torch.float32, device="cuda")
        st = L.kvq_decode_attn_packed_ex(kvq._dptr(table.table), n, H, Hq, D, 4, kvq._dptr(q3[:n].contiguous()),
                                         ctypes.c_float(0.088), kvq._dptr(out), kvq._dptr(ws), ws.numel(), algo, None)
        torch.cuda.synchronize()
        assert st == 0 and kvq.attn_error_word(ws) == 0, algo
        return out.cpu().numpy()

    int4 = kvq.RequestTable(kc4, vc4, torch.device("cuda"))
    plain = call(int4, 2, kvq.ATTN_MMA)
    assert np.array_equal(call(int4, 2, kvq.ATTN_MMA | kvq.ATTN_NVFP4), plain)
    assert np.array_equal(call(int4, 2, kvq.ATTN_AUTO | kvq.ATTN_NVFP4), plain)
    mixed = kvq.RequestTable(kc4[:1] + kc + kc4[1:], vc4[:1] + vc + vc4[1:], torch.device("cuda"))
    flagged = call(mixed, 3, kvq.ATTN_MMA | kvq.ATTN_NVFP4)
    assert np.array_equal(flagged, call(mixed, 3, kvq.ATTN_MMA_GENERAL | kvq.ATTN_NVFP4))
    ref = lambda b, ok_, ov_: O.attention_f32(bf16_bits(q3[b].cpu()), O.decode_f32(ok_, 4),  # noqa: E731
                                              O.decode_f32(ov_, 4), 0.088)
    for b, (ok_, ov_) in enumerate([(oks4[0], ovs4[0]), (oks[0], ovs[0]), (oks4[1], ovs4[1])]):
        P.assert_attention_close(flagged[b], ref(b, ok_, ov_), f"mixed table, request {b}")
    for b in range(2):
        P.assert_attention_close(plain[b], ref(b, oks4[b], ovs4[b]), f"INT4 table, request {b}")


def test_sparse_later_loop_without_the_nvfp4_flag_refuses_nvfp4():
    """The tensor-core sparse later loop called without KVQ_ATTN_NVFP4: the request
    holding NVFP4 loops is refused (NaN, bit 64), the INT4 request beside it agrees
    with the same call with the flag (within the attention tolerance: without the
    flag it runs the INT4 kernel, with it the NVFP4-capable one)."""
    H, Hq = 8, 32
    _, kc, vc, oks, ovs, q = _nvfp4_requests([300], Hq, 710)
    _, kc4, vc4, oks4, ovs4, _ = _nvfp4_requests([200], Hq, 711, (I4, I4, I4, I4))
    table = kvq.RequestTable(kc + kc4, vc + vc4, torch.device("cuda"))
    q2 = torch.randn((2, Hq, D), generator=torch.Generator().manual_seed(712)).to(torch.bfloat16).cuda()
    st = kvq.kvq_sparse_ref_state(table, q2, 2, H, 64, 300)
    L = kvq.lib()
    outs = []
    for algo in (kvq.ATTN_MMA, kvq.ATTN_MMA | kvq.ATTN_NVFP4):
        ws = torch.zeros(kvq.kvq_sparse_decode_workspace_bytes(2, H, Hq, D, 300), dtype=torch.uint8, device="cuda")
        out = torch.empty((2, Hq, D), dtype=torch.float32, device="cuda")
        sel = st.sel_idx.contiguous()
        rc = L.kvq_sparse_decode_attn_ex(kvq._dptr(table.table), 2, H, Hq, D, 4, kvq._dptr(q2), ctypes.c_float(0.088),
                                         64, 300, kvq._dptr(sel), kvq._dptr(st.mass), kvq._dptr(st.o_ref),
                                         kvq._dptr(st.c_ref), kvq._dptr(out), kvq._dptr(ws), ws.numel(), algo, None)
        torch.cuda.synchronize()
        assert rc == 0
        outs.append((out.cpu().numpy(), kvq.attn_error_word(ws)))
    (o_no, e_no), (o_nv, e_nv) = outs
    assert e_no & 64 and np.all(np.isnan(o_no[0])) and e_nv == 0 and not np.any(np.isnan(o_nv))
    P.assert_attention_close(o_no[1], o_nv[1], "INT4 request")


def test_nvfp4_sparse_decode():
    """Sparse decode attention (FlashLoop RFC §3.2) over NVFP4 residual loops."""
    lengths = [1000, 300]
    Hq = 32
    H, kc, vc, oks, ovs, q = _nvfp4_requests(lengths, Hq, 600)
    table = kvq.RequestTable(kc, vc, torch.device("cuda"))
    scale = 1.0 / math.sqrt(D)
    st = kvq.kvq_sparse_ref_state(table, q.cuda(), 2, H, 128, max(lengths))
    q4 = torch.randn((len(lengths), Hq, D), generator=torch.Generator().manual_seed(601)).to(torch.bfloat16)
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")  # the per-key kernel
    out = kvq.kvq_sparse_decode_attn(table, q4.cuda(), 4, H, st, workspace=ws).cpu().numpy()
    wsb = torch.zeros(kvq.kvq_sparse_decode_workspace_bytes(len(lengths), H, Hq, D, max(lengths)), dtype=torch.uint8,
                      device="cuda")  # the key-masked tensor-core attention
    out_tc = kvq.kvq_sparse_decode_attn(table, q4.cuda(), 4, H, st, workspace=wsb, algo=kvq.ATTN_MMA).cpu().numpy()
    torch.cuda.synchronize()
    assert kvq.attn_error_word(st.workspace) == 0 and kvq.attn_error_word(ws) == 0 and kvq.attn_error_word(wsb) == 0
    sel, mass, o_ref, c_ref = (t.cpu().numpy() for t in (st.sel_idx, st.mass, st.o_ref, st.c_ref))
    for b, T in enumerate(lengths):
        S = sel[b][:, :min(128, T)]
        kf2, vf2 = O.decode_f32(oks[b], 2), O.decode_f32(ovs[b], 2)
        P.assert_attention_close(o_ref[b], O.attention_f32(bf16_bits(q[b]), kf2, vf2, scale), f"O_ref req {b}")
        ref = O.sparse_decode(bf16_bits(q4[b]), O.decode_f32(oks[b], 4), O.decode_f32(ovs[b], 4), scale, S,
                              mass[b].astype(np.float64), o_ref[b].astype(np.float64), c_ref[b].astype(np.float64))
        P.assert_attention_close(out[b], ref, f"sparse req {b}")
        P.assert_attention_close(out_tc[b], ref, f"sparse req {b}, tensor-core path")
