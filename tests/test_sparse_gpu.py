"""Sparse decode attention over the packed chains (FlashLoop RFC, vllm-rlt
issue #156, §3.2), through the C ABI, against the oracle on the same packed
data: the reference state at loop 2 (selection, mass, full output, selected
contribution) and the corrected output of loops 3 and 4.

The selection is decided in floating point on both sides (FP32 on the GPU,
float64 in the oracle), so keys whose probabilities tie with the k-th one to
within rounding may differ; the test checks the GPU selection against the
oracle's probabilities (every selected key at least, every other key at most,
the k-th probability up to 1e-5 relative) and then compares mass, C_ref and
the later-loop output computed from that selection. Each later loop runs on
both kernels: the per-key gather (a 16-byte workspace) and the key-masked
tensor-core attention."""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from quantized_cross_loop_gb300 import kvq
from quantized_cross_loop_gb300 import workloads as W
from quantized_cross_loop_gb300.workloads import bf16_bits

from tests import pathrun as P

pytestmark = pytest.mark.gpu

H, D = 8, 128
PATHS = ("per_key", "tensor_core")


def _decode(table, q, depth, st, path, Hq):
    """A later loop on one of the two kernels; returns (out, error word)."""
    if path == "per_key":
        ws, algo = torch.zeros(16, dtype=torch.uint8, device="cuda"), kvq.ATTN_SIMT
    else:
        n = kvq.kvq_sparse_decode_workspace_bytes(q.shape[0], H, Hq, D, st.max_tokens)
        ws, algo = torch.zeros(n, dtype=torch.uint8, device="cuda"), kvq.ATTN_MMA
    out = kvq.kvq_sparse_decode_attn(table, q.cuda(), depth, H, st, workspace=ws, algo=algo)
    torch.cuda.synchronize()
    return out.cpu().numpy(), kvq.attn_error_word(ws)


def _setup(Ts, sparse, Hq=32, seed=0):
    reqs, kc, vc, oks, ovs = [], [], [], [], []
    for b, T in enumerate(Ts):
        spec = W.ConfigSpec("sp", seed + b, 1, max(T, 1), H, D, Hq, 4, 0.1,
                            (1.0, 1.0, 0.5, 0.25) if sparse else (1.0, 1.0, 1.0, 1.0))
        r = W.make_request(spec, 0, 0, "cpu", T=T, sparse=sparse)
        k, v = P.gpu_chains(r)
        kc.append(k)
        vc.append(v)
        act = [None if a is None else a.numpy().astype(np.int32) for a in r.active]
        oks.append(O.encode_chain(O.KIND_K, [bf16_bits(x) for x in r.xk], act))
        ovs.append(O.encode_chain(O.KIND_V, [bf16_bits(x) for x in r.xv], act))
        reqs.append(r)
    table = kvq.RequestTable(kc, vc, torch.device("cuda"))
    g = torch.Generator().manual_seed(seed + 100)
    qs = [torch.randn((len(Ts), Hq, D), generator=g).to(torch.bfloat16) for _ in range(3)]  # loops 2, 3, 4
    return table, reqs, oks, ovs, qs


def _logits64(q_bits, kf, hq, g, scale):
    return np.asarray(kf, np.float64)[:, hq // g, :] @ O.bf16_bits_to_f32(q_bits[hq]).astype(np.float64) * scale


def _check_selection(sel, q_bits, kf, Hq, g, K, scale):
    T = kf.shape[0]
    for hq in range(Hq):
        s = _logits64(q_bits, kf, hq, g, scale)
        S = sel[hq][:K]
        assert len(S) == K and np.all(np.diff(S) > 0) and (K == 0 or (S[0] >= 0 and S[-1] < T))
        if K == 0 or K == T:
            assert K == 0 or np.array_equal(S, np.arange(T))
            continue
        kth = np.sort(s)[::-1][K - 1]
        tol = 1e-5 * max(1.0, abs(kth))
        mask = np.zeros(T, bool)
        mask[S] = True
        assert np.all(s[mask] >= kth - tol), f"head {hq}: a selected key below the k-th"
        assert np.all(s[~mask] <= kth + tol), f"head {hq}: an unselected key above the k-th"


@pytest.mark.parametrize("Ts,sparse,n_select,Hq", [
    ([300, 1000], True, 64, 32),
    ([4096], False, 1024, 32),
    ([777, 64, 1], True, 100, 64),
    ([200], False, 500, 32),  # more than T: every key
    ([1000, 300], True, 10, 32),  # at most max_tokens / 64 keys: C_ref gathered key by key
    ([12300, 40], False, 400, 32),  # beyond the staged length: keys re-read, C_ref key by key
])
def test_sparse_reference_and_later_loops(Ts, sparse, n_select, Hq):
    table, reqs, oks, ovs, qs = _setup(Ts, sparse, Hq, seed=sum(Ts) + n_select)
    g = Hq // H
    scale = 1.0 / math.sqrt(D)
    max_tokens = max(Ts)
    st = kvq.kvq_sparse_ref_state(table, qs[0].cuda(), 2, H, n_select, max_tokens)
    torch.cuda.synchronize()
    assert kvq.attn_error_word(st.workspace) == 0
    sel, mass, o_ref, c_ref = (t.cpu().numpy() for t in (st.sel_idx, st.mass, st.o_ref, st.c_ref))
    outs = {}
    for path in PATHS:
        for depth, q in ((3, qs[1]), (4, qs[2])):
            outs[path, depth], err = _decode(table, q, depth, st, path, Hq)
            assert err == 0, path
    for b, T in enumerate(Ts):
        K = min(n_select, T)
        assert np.all(sel[b][:, K:] == -1)
        kf2, vf2 = O.decode_f32(oks[b], 2), O.decode_f32(ovs[b], 2)
        qb = bf16_bits(qs[0][b])
        _check_selection(sel[b], qb, kf2, Hq, g, K, scale)
        # the oracle's state on the GPU's selection
        S = sel[b][:, :K]
        m_o, c_o, o_o = np.zeros(Hq), np.zeros((Hq, D)), np.zeros((Hq, D))
        for hq in range(Hq):
            s = _logits64(qb, kf2, hq, g, scale)
            p = np.exp(s - s.max())
            p /= p.sum()
            m_o[hq] = p[S[hq]].sum()
            c_o[hq] = p[S[hq]] @ np.asarray(vf2, np.float64)[S[hq], hq // g, :]
            o_o[hq] = p @ np.asarray(vf2, np.float64)[:, hq // g, :]
        assert np.max(np.abs(mass[b] - m_o)) < 1e-4
        P.assert_attention_close(c_ref[b], c_o, f"C_ref req {b}")
        P.assert_attention_close(o_ref[b], o_o, f"O_ref req {b}")
        # later loops from the GPU state
        for depth, q in ((3, qs[1]), (4, qs[2])):
            kf, vf = O.decode_f32(oks[b], depth), O.decode_f32(ovs[b], depth)
            ref = O.sparse_decode(bf16_bits(q[b]), kf, vf, scale, S, mass[b].astype(np.float64),
                                  o_ref[b].astype(np.float64), c_ref[b].astype(np.float64))
            for path in PATHS:
                P.assert_attention_close(outs[path, depth][b], ref, f"req {b} depth {depth} {path}")
                if K == T:  # every key kept: plain dense attention at this depth
                    dense = O.attention_f32(bf16_bits(q[b]), kf, vf, scale)
                    P.assert_attention_close(outs[path, depth][b], dense, f"dense req {b} depth {depth} {path}")


@pytest.mark.parametrize("n_select", [10, 64, 70])
def test_sparse_selection_breaks_exact_ties_by_position(n_select):
    """Keys with exactly equal logits: tokens 64-127 of each KV head share one K
    row (a constant K group, so equal codes and parameters), built to outscore
    every other key for each of the head's query heads. The selection takes the
    lowest positions among them (RFC §3.2 top-k with the position tie-break);
    beyond 64 keys it takes the whole tied group, then the best of the rest, as
    the oracle's logits rank them."""
    T, Hq = 256, 32
    g = Hq // H
    gen = torch.Generator().manual_seed(77)
    q = torch.randn((1, Hq, D), generator=gen).to(torch.bfloat16)
    xk = torch.randn((T, H, D), generator=gen) * 0.5
    xv = torch.randn((T, H, D), generator=gen)
    for h in range(H):  # the tied row: along the sum of the head's queries
        xk[64:128, h] = 0.25 * q[0, g * h:g * h + g].float().sum(0)
    xk, xv = xk.to(torch.bfloat16), xv.to(torch.bfloat16)
    kc = [kvq.kvq_encode_base(xk.cuda(), kvq.KVQ_K)]
    vc = [kvq.kvq_encode_base(xv.cuda(), kvq.KVQ_V)]
    table = kvq.RequestTable([kc], [vc], torch.device("cuda"))
    st = kvq.kvq_sparse_ref_state(table, q.cuda(), 1, H, n_select, T)
    torch.cuda.synchronize()
    assert kvq.attn_error_word(st.workspace) == 0
    sel = st.sel_idx.cpu().numpy()[0]
    ok = O.encode_chain(O.KIND_K, [bf16_bits(xk)], [None])
    kf = O.decode_f32(ok, 1)
    qb = bf16_bits(q[0])
    for hq in range(Hq):
        s64 = _logits64(qb, kf, hq, g, 1.0 / math.sqrt(D))
        assert np.all(s64[64:128] == s64[64]) and s64[64] > np.delete(s64, np.arange(64, 128)).max()
        if n_select <= 64:
            assert np.array_equal(sel[hq], np.arange(64, 64 + n_select)), hq
            continue
        S = sel[hq]
        assert len(S) == n_select and np.all(np.diff(S) > 0) and np.all(np.isin(np.arange(64, 128), S)), hq
        rest = np.delete(np.arange(T), np.arange(64, 128))
        picked = np.isin(rest, S)
        tol = 1e-5 * max(1.0, float(np.abs(s64).max()))  # FP32 logits on the GPU, float64 here
        assert picked.sum() == n_select - 64 and s64[rest[picked]].min() >= s64[rest[~picked]].max() - tol, hq


def test_sparse_refuses_segments_and_bad_selections():
    table, reqs, oks, ovs, qs = _setup([100, 100], False, 32, seed=9)
    seg = tuple(torch.randn((n, H, D)).to(torch.bfloat16).cuda() for n in (2, 2, 0, 0))
    table2 = kvq.RequestTable([table._keep[0][0], table._keep[0][1]], [table._keep[1][0], table._keep[1][1]],
                              torch.device("cuda"), segments=[seg, None])
    st = kvq.kvq_sparse_ref_state(table2, qs[0].cuda(), 2, H, 16, 100)
    torch.cuda.synchronize()
    assert kvq.attn_error_word(st.workspace) != 0
    assert np.all(np.isnan(st.mass.cpu().numpy()[0])) and not np.any(np.isnan(st.mass.cpu().numpy()[1]))
    # a later loop refuses the request with segments on both kernels
    for path in PATHS:
        out, err = _decode(table2, qs[1], 3, st, path, 32)
        assert err & 1 and np.all(np.isnan(out[0])) and not np.any(np.isnan(out[1])), path
    # a corrupted selection (position past the request) is flagged, not read
    st = kvq.kvq_sparse_ref_state(table, qs[0].cuda(), 2, H, 16, 100)
    st.sel_idx[1, 0, 3] = 5000
    for path in PATHS:
        out, err = _decode(table, qs[1], 3, st, path, 32)
        assert err & 32 and not np.any(np.isnan(out)), path


def test_sparse_refuses_requests_longer_than_max_tokens():
    """max_tokens below one request's length: that request is refused (NaN, bit 1)
    by the reference pass and by both later-loop kernels, which read no key mask
    or logit row past its end; the other request is unaffected."""
    table, reqs, oks, ovs, qs = _setup([100, 200], False, 32, seed=31)
    st = kvq.kvq_sparse_ref_state(table, qs[0].cuda(), 2, H, 16, 150)
    torch.cuda.synchronize()
    assert kvq.attn_error_word(st.workspace) & 1
    mass = st.mass.cpu().numpy()
    assert np.all(np.isnan(mass[1])) and not np.any(np.isnan(mass[0]))
    scale = 1.0 / math.sqrt(D)
    S = st.sel_idx.cpu().numpy()[0][:, :16]
    ref = O.sparse_decode(bf16_bits(qs[1][0]), O.decode_f32(oks[0], 3), O.decode_f32(ovs[0], 3), scale, S,
                          mass[0].astype(np.float64), st.o_ref.cpu().numpy()[0].astype(np.float64),
                          st.c_ref.cpu().numpy()[0].astype(np.float64))
    for path in PATHS:
        out, err = _decode(table, qs[1], 3, st, path, 32)
        assert err & 1 and np.all(np.isnan(out[1])), path
        P.assert_attention_close(out[0], ref, f"request 0 {path}")


def test_sparse_empty_selection_and_path_choice():
    """n_select = 0: the later loop returns O_ref - C_ref on both kernels. The
    tensor-core path asked for explicitly with a small workspace is an error;
    AUTO with a small workspace takes the per-key kernel."""
    table, reqs, oks, ovs, qs = _setup([300, 65], True, 32, seed=21)
    st = kvq.kvq_sparse_ref_state(table, qs[0].cuda(), 2, H, 0, 300)
    torch.cuda.synchronize()
    expect = (st.o_ref - st.c_ref).cpu().numpy()
    for path in PATHS:
        out, err = _decode(table, qs[1], 4, st, path, 32)
        assert err == 0 and np.array_equal(out, expect), path
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError):
        kvq.kvq_sparse_decode_attn(table, qs[1].cuda(), 4, H, st, workspace=small, algo=kvq.ATTN_MMA)
    kvq.kvq_sparse_decode_attn(table, qs[1].cuda(), 4, H, st, workspace=small)
    torch.cuda.synchronize()
    assert kvq.attn_error_word(small) == 0


def test_sparse_auto_takes_the_gather_for_small_selections():
    """With a workspace large enough for the key-masked path, AUTO gathers a
    selection of at most max_tokens / 64 keys per query head key by key (the
    masked attention would still read every tile) and attends larger ones
    through key masks: AUTO's output equals that kernel's bit for bit."""
    table, reqs, oks, ovs, qs = _setup([1000, 777], True, 32, seed=5)
    n = kvq.kvq_sparse_decode_workspace_bytes(2, H, 32, D, 1000)
    for n_select, path in ((15, "per_key"), (16, "tensor_core"), (120, "tensor_core")):
        st = kvq.kvq_sparse_ref_state(table, qs[0].cuda(), 2, H, n_select, 1000)
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
        auto = kvq.kvq_sparse_decode_attn(table, qs[1].cuda(), 4, H, st, workspace=ws).cpu().numpy()
        assert kvq.attn_error_word(ws) == 0
        ref, err = _decode(table, qs[1], 4, st, path, 32)
        assert err == 0 and np.array_equal(auto, ref), (n_select, path)
