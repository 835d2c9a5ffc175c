"""Pins for the CPU oracle: facts fixed by the pages, by IEEE-754 and by
mathematics, checked without reusing the oracle's own formulas.

Page titles used below: "FlashLoop RFC" = "[RFC]: FlashLoop integration —
token-sparse prefill, sparse decode attention, and KV residual quantization"
(vllm-rlt issue #156); "codec PR" = "INT4 KV packing/unpacking and cross-loop
residual reconstruction" (vllm-rlt pull #166).
"""

from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests import reader_bound as RB

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bf16(a) -> np.ndarray:
    """float values -> BF16 bits via torch's cast (a library routine)."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f32(bits) -> np.ndarray:
    return O.bf16_bits_to_f32(bits)


def f16_to_f32(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def unpack(codes: np.ndarray) -> np.ndarray:
    """uint8 [H, n, D/2] -> int codes [n, H, D]: the low nibble holds the even channel."""
    H, n, half = codes.shape
    out = np.empty((n, H, 2 * half), dtype=np.int64)
    out[:, :, 0::2] = np.transpose(codes & 0x0F, (1, 0, 2))
    out[:, :, 1::2] = np.transpose(codes >> 4, (1, 0, 2))
    return out


# ---------------------------------------------------------------- IEEE rounding helpers


def _sample_f32_bits(n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    r = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    # add every pattern whose low 16 bits sit at or next to a rounding tie, and special values
    hi = rng.integers(0, 2**16, size=4096, dtype=np.uint64).astype(np.uint32) << 16
    low = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1000, 0x0FFF, 0x1001, 0x2000, 0x3000],
                   dtype=np.uint32)
    ties = (hi[:, None] | low[None, :]).ravel()
    special = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7F7FFFFF, 0x477FEFFF, 0x477FF000, 0x477FF001,
                        0x38800000, 0x387FFFFF, 0x33800000, 0x33000000, 0x33000001, 0x00000001, 0x80000001],
                       dtype=np.uint32)
    # the whole binary16 subnormal/normal boundary region, densely
    dense = (np.arange(0x33000000, 0x38900000, 97, dtype=np.uint64)).astype(np.uint32)
    return np.concatenate([r, ties, special, dense])


def test_f32_to_f16_matches_numpy_cast():
    bits = _sample_f32_bits(1 << 22, 1)
    x = bits.view(np.float32)
    ours = O.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(ours[nan].view(np.float16)))


def test_f16_to_f32_exhaustive():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = O.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert np.all(np.isnan(ours[nan]))


def test_f32_to_bf16_matches_torch_cast():
    bits = _sample_f32_bits(1 << 22, 2)
    x = bits.view(np.float32)
    ours = O.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(f32(ours[nan])))


# ---------------------------------------------------------------- the INT4 group quantiser


def _k_stream_of_columns(cols: np.ndarray):
    """Encode columns cols[:, j] (each one K group over rows) as a K base stream."""
    n, m = cols.shape
    assert m % 2 == 0
    x = bf16(cols.reshape(n, 1, m))
    return x, O.encode(O.KIND_K, x)


def _check_group_brute(xs: np.ndarray, codes: np.ndarray, min16: int, scale16: int):
    """Exact-rational check of one group (xs: FP32 values of the BF16 inputs).

    FlashLoop RFC §3.3: scale = (max - min)/15, code = rounded/clipped
    (x - min)/scale; codec PR review by 0z5a: codes come from the FP32 scale,
    the FP16 metadata is rounded afterwards.
    """
    mn, mx = float(np.min(xs)), float(np.max(xs))
    assert codes.min() >= 0 and codes.max() <= 15
    assert min16 == int(np.float16(np.float32(mn)).view(np.uint16))
    if mx == mn:  # constant group: explicit, every code 0, scale stored as 0
        assert np.all(codes == 0) and scale16 == 0
        return
    s32 = np.float32(np.float32(np.float32(mx) - np.float32(mn)) / np.float32(15.0))
    assert scale16 == int(np.float16(s32).view(np.uint16))
    S = Fraction(float(s32))
    slack = Fraction(1, 1 << 19)  # FP32 rounding of (x - min) and of the ratio, in units of the scale
    for x, c in zip(xs.tolist(), codes.tolist()):
        r = (Fraction(x) - Fraction(mn)) / S
        dist = abs(r - c)
        assert dist <= Fraction(1, 2) + slack, (x, c, float(r))
        for c2 in range(16):  # no other level is clearly closer
            assert abs(r - c2) >= dist - 2 * slack, (x, c, c2)
    # the group's minimum maps to code 0 and its maximum to code 15
    assert codes[int(np.argmin(xs))] == 0
    assert codes[int(np.argmax(xs))] == 15


@pytest.mark.parametrize("n", [1, 2, 3, 5, 17, 64])
def test_quantiser_brute_force_random(n):
    rng = np.random.default_rng(100 + n)
    for trial in range(20):
        cols = rng.standard_normal((n, 4)).astype(np.float32) * rng.choice([1e-3, 0.1, 1.0, 30.0])
        cols[:, 3] = cols[0, 3]  # one constant column
        x, s = _k_stream_of_columns(cols)
        c = unpack(s.codes)[:, 0, :]
        xs = f32(x)[:, 0, :]
        for j in range(4):
            _check_group_brute(xs[:, j], c[:, j], int(s.mins[0, 0, j]), int(s.scales[0, 0, j]))


def test_quantiser_ties_round_half_even():
    # min 0 and max 15 make the scale exactly 1, so (x - min)/scale is exact
    col = np.array([0.0, 15.0, 0.5, 1.5, 2.5, 3.5, 6.5, 7.5, 14.5, 13.5], dtype=np.float32)
    cols = np.stack([col, col], axis=1)
    _, s = _k_stream_of_columns(cols)
    c = unpack(s.codes)[:, 0, 0]
    assert c.tolist() == [0, 15, 0, 2, 2, 4, 6, 8, 14, 14]


def test_codes_use_fp32_scale_not_fp16_scale():
    """Codec PR review by 0z5a: codes come from the FP32 scale before the FP16
    metadata is rounded. Find a BF16 value whose code differs under the two."""
    cand = None
    for mx in (1.0078125, 1.0234375, 1.3671875, 1.6328125, 1.8828125, 2.0625, 3.8125):
        mx = np.float32(mx)
        s32 = np.float32(mx / np.float32(15.0))
        s16 = np.float32(np.float16(s32))
        if s16 == s32:
            continue
        vals = torch.arange(1, 1 << 15, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float().numpy()
        vals = vals[(vals > 0) & (vals < mx)]
        r32 = np.rint((vals / s32).astype(np.float32))
        r16 = np.rint((vals / s16).astype(np.float32))
        hit = np.nonzero(r32 != r16)[0]
        if hit.size:
            cand = (mx, np.float32(vals[hit[0]]), int(r32[hit[0]]), int(r16[hit[0]]))
            break
    assert cand is not None
    mx, v, code32, code16 = cand
    col = np.array([0.0, mx, v, v], dtype=np.float32)
    _, s = _k_stream_of_columns(np.stack([col, col], axis=1))
    c = unpack(s.codes)[2, 0, 0]
    assert c == code32 and c != code16


def test_constant_group_decodes_to_min16():
    # FlashLoop RFC §3.3 and §9: constant groups are defined explicitly (no division by zero)
    cols = np.full((64, 2), 3.140625, dtype=np.float32)
    x, s = _k_stream_of_columns(cols)
    assert np.all(unpack(s.codes) == 0) and np.all(s.scales == 0)
    out = O.reconstruct([s], 1)
    expect = bf16(f16_to_f32(s.mins[0, 0, 0]))
    assert np.all(out == expect[()])
    v = O.encode(O.KIND_V, bf16(np.full((3, 2, 128), -0.75, dtype=np.float32)))
    assert np.all(v.scales == 0)
    assert np.all(O.reconstruct([v], 1) == bf16(np.float32(-0.75))[()])


@pytest.mark.parametrize("seed", range(3))
def test_round_trip_bound(seed):
    """|x - decode| <= scale/2 plus the FP16 metadata and BF16 output roundings."""
    rng = np.random.default_rng(seed)
    T, H, D = 70, 2, 96  # a partial K row group (6 rows) and a partial V channel group (32)
    x = bf16(rng.standard_normal((T, H, D)) * 2.0)
    xf = f32(x).astype(np.float64)
    for kind in (O.KIND_K, O.KIND_V):
        s = O.encode(kind, x)
        dec = f32(O.reconstruct([s], 1)).astype(np.float64)
        for t in range(T):
            for h in range(H):
                for d in range(D):
                    if kind == O.KIND_K:
                        rows = slice((t // 64) * 64, min((t // 64) * 64 + 64, T))
                        grp = xf[rows, h, d]
                        p = (h, t // 64, d)
                    else:
                        c0 = (d // 64) * 64
                        grp = xf[t, h, c0:min(c0 + 64, D)]
                        p = (h, t, d // 64)
                    mn, mx = grp.min(), grp.max()
                    s32 = float(np.float32(np.float32(mx - mn) / np.float32(15)))
                    m16 = float(f16_to_f32(s.mins[p]))
                    sc16 = float(f16_to_f32(s.scales[p]))
                    bound = (s32 / 2 * (1 + 2**-18) + abs(mn - m16) + 15 * abs(s32 - sc16)
                             + 2.0 ** (math.frexp(abs(dec[t, h, d]) or 1e-30)[1] - 9) + 1e-30)
                    assert abs(xf[t, h, d] - dec[t, h, d]) <= bound, (kind, t, h, d)


# ---------------------------------------------------------------- group geometry and packing


@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 129, 1000])
def test_group_boundaries_and_partial_tails(T):
    """K groups hold <= 64 consecutive rows per (head, channel); V groups 64
    channels per (row, head); tails hold only their true rows (codec PR, Purpose)."""
    rng = np.random.default_rng(T)
    H, D = 2, 128
    x = bf16(rng.standard_normal((T, H, D)))
    xf = f32(x)
    k = O.encode(O.KIND_K, x)
    assert k.mins.shape == (H, -(-T // 64), D)
    for g in range(-(-T // 64)):
        rows = xf[g * 64:min(g * 64 + 64, T)]
        mn = rows.min(axis=0)  # [H, D]
        assert np.array_equal(k.mins[:, g, :], mn.astype(np.float16).view(np.uint16))
        mx = rows.max(axis=0)
        s32 = ((mx - mn).astype(np.float32) / np.float32(15)).astype(np.float32)
        s32[mx == mn] = 0
        assert np.array_equal(k.scales[:, g, :], s32.astype(np.float16).view(np.uint16))
    v = O.encode(O.KIND_V, x)
    assert v.mins.shape == (H, T, 2)
    for c in range(2):
        grp = xf[:, :, c * 64:(c + 1) * 64]
        assert np.array_equal(v.mins[:, :, c], grp.min(axis=2).T.astype(np.float16).view(np.uint16))


def test_v_partial_channel_group():
    rng = np.random.default_rng(7)
    x = bf16(rng.standard_normal((5, 1, 80)))
    xf = f32(x)
    v = O.encode(O.KIND_V, x)
    assert v.mins.shape == (1, 5, 2)
    assert np.array_equal(v.mins[0, :, 1], xf[:, 0, 64:80].min(axis=1).astype(np.float16).view(np.uint16))


def test_nibble_order_fixture():
    gold = json.load(open(os.path.join(GOLD, "nibble_order.json")))
    vc = gold["v_case"]
    v = O.encode(O.KIND_V, bf16(np.array(vc["x"], dtype=np.float32).reshape(1, 1, 4)))
    assert v.codes.ravel().tolist() == vc["bytes"]
    assert unpack(v.codes).ravel().tolist() == vc["codes"]
    kc = gold["k_case"]
    k = O.encode(O.KIND_K, bf16(np.array(kc["x"], dtype=np.float32).reshape(4, 1, 2)))
    assert k.codes.ravel().tolist() == kc["bytes_by_row"]


def test_head_major_plane_layout():
    """Byte (h, row, k) holds channels 2k, 2k+1 of (row, head h)."""
    T, H, D = 3, 2, 4
    x = np.zeros((T, H, D), dtype=np.float32)
    x[:, :, 0] = 0.0
    x[:, :, 1] = 15.0  # each V group: min 0 (channel 0), max 15 (channel 1), scale 1
    x[1, 1, 2] = 7.0
    x[2, 0, 3] = 9.0
    v = O.encode(O.KIND_V, bf16(x))
    assert v.codes.shape == (H, T, 2)
    assert v.codes[1, 1, 1] == 7 and v.codes[0, 2, 1] == 9 << 4
    assert np.all(v.codes[:, :, 0] == 0xF0)


# ---------------------------------------------------------------- residual chains


def test_residual_subtracts_reconstructed_predecessor():
    """FlashLoop RFC §3.3 worked example: the residual is X[2] - X̂[1]; a raw
    difference X[2] - X[1] would keep the first loop's error. With X2 == X1 the
    raw difference is zero, while the right residual cancels most of the base error."""
    rng = np.random.default_rng(11)
    T, H, D = 128, 2, 128
    x1 = bf16(rng.standard_normal((T, H, D)) * 3.0)
    for kind in (O.KIND_K, O.KIND_V):
        ks = O.encode_chain(kind, [x1, x1], [None, None])
        e1 = np.abs(f32(O.reconstruct(ks, 1)) - f32(x1)).max()
        e2 = np.abs(f32(O.reconstruct(ks, 2)) - f32(x1)).max()
        assert e1 > 0.05
        assert e2 < e1 / 6, (kind, e1, e2)
        # the stored residual is exactly the quantisation of RN_bf16(X2 - X̂1)
        xhat1 = f32(O.reconstruct(ks, 1))
        delta = bf16(f32(x1) - xhat1)
        ref = O.encode(kind, delta)
        assert np.array_equal(ref.codes, ks[1].codes)
        assert np.array_equal(ref.mins, ks[1].mins) and np.array_equal(ref.scales, ks[1].scales)


def _offset_chain(T, H, D, seed):
    rng = np.random.default_rng(seed)
    xs = [rng.standard_normal((T, H, D)).astype(np.float32)]
    for r in range(1, 4):
        # a positive drift, so every residual group has a nonzero FP16 minimum
        xs.append(xs[-1] + 0.25 + 0.1 * np.abs(rng.standard_normal((T, H, D))).astype(np.float32))
    return [bf16(x) for x in xs]


def test_loop4_read_example_inheritance():
    """FlashLoop RFC §3.1 eight-token example and §3.3 loop-4 read resolution:
    an absent residual means inheritance, not an INT4 code 0."""
    gold = json.load(open(os.path.join(GOLD, "loop4_read_example.json")))
    T = gold["T"]
    act = {int(r): np.array(v, dtype=np.int32) - 1 for r, v in gold["active_1based"].items()}
    xs = _offset_chain(T, 2, 128, 5)
    actives = [None, None, act[3], act[4]]
    for kind in (O.KIND_K, O.KIND_V):
        ks = O.encode_chain(kind, xs, actives)
        assert ks[2].n == 4 and ks[3].n == 2
        assert np.all(f16_to_f32(ks[3].mins) > 0)  # a code-0 read would add this minimum
        rec = {d: O.reconstruct(ks, d) for d in range(1, 5)}
        for tok1, loops in gold["loop4_read_1based"].items():
            t = int(tok1) - 1
            last = max(loops)
            # the value changes at each listed loop and never after the last one
            for d in range(2, 5):
                changed = not np.array_equal(rec[d][t], rec[d - 1][t])
                assert changed == (d in loops), (kind, tok1, d)
            assert np.array_equal(rec[4][t], rec[last][t])
        # every token outside A4 keeps its depth-3 bits at depth 4
        for t in range(T):
            if t not in act[4]:
                assert np.array_equal(rec[4][t], rec[3][t])


def test_dense_equals_full_sparse():
    T, H, D = 200, 2, 128
    xs = _offset_chain(T, H, D, 9)
    full = np.arange(T, dtype=np.int32)
    for kind in (O.KIND_K, O.KIND_V):
        a = O.encode_chain(kind, xs, [None] * 4)
        b = O.encode_chain(kind, xs, [None, full, full, full])
        for sa, sb in zip(a, b):
            assert np.array_equal(sa.codes, sb.codes)
            assert np.array_equal(sa.mins, sb.mins) and np.array_equal(sa.scales, sb.scales)
        assert np.array_equal(O.reconstruct(a, 4), O.reconstruct(b, 4))


def test_sparse_k_groups_follow_compact_rows():
    """Codec PR review by 0z5a: sparse K groups run over compact rows, so one
    group can mix distant logical positions."""
    T, H, D = 300, 1, 128
    xs = _offset_chain(T, H, D, 13)
    rng = np.random.default_rng(3)
    a = np.sort(rng.choice(T, 130, replace=False)).astype(np.int32)
    ks = O.encode_chain(O.KIND_K, xs[:2] + [xs[2]], [None, None, a])
    s = ks[2]
    assert s.mins.shape == (H, 3, D)  # ceil(130/64) groups: 64, 64, 2 rows
    pred = f32(O.reconstruct(ks, 2))
    delta = f32(bf16(f32(xs[2])[a] - pred[a]))  # [130, H, D]
    for g, rows in enumerate([slice(0, 64), slice(64, 128), slice(128, 130)]):
        assert np.array_equal(s.mins[:, g, :], delta[rows].min(axis=0).astype(np.float16).view(np.uint16))


def _tile_chain(T, H, D, seed, drop_tile=2):
    """A sparse loop-3 chain whose active set misses one whole 64-token tile."""
    xs = _offset_chain(T, H, D, seed)
    rng = np.random.default_rng(seed + 1)
    a = np.sort(rng.choice(T, T // 2, replace=False)).astype(np.int32)
    a = a[(a // 64) != drop_tile]
    return xs, a


def test_tile_k_groups_hold_one_logical_tile():
    """Codec PR review by 0z5a (group ownership vs pages): under tile grouping a
    sparse K group holds exactly the stored rows of one 64-token logical tile;
    its FP16 min and scale are those of that group's residuals (numpy min/max,
    FP32 division by 15, then the FP16 cast), and a tile with no stored row keeps
    +0 min and +0 scale."""
    T, H, D = 300, 2, 128
    xs, a = _tile_chain(T, H, D, 21)
    ks = O.encode_chain(O.KIND_K, xs[:3], [None, None, a], kgroup=O.KGROUP_TILE)
    s = ks[2]
    assert s.mins.shape == (H, 5, D)  # ceil(300/64) logical tiles, whatever |a| is
    pred = f32(O.reconstruct(ks, 2))
    delta = f32(bf16(f32(xs[2])[a] - pred[a]))  # [n, H, D] in compact order
    codes = unpack(s.codes)
    for k in range(5):
        rows = np.nonzero(a // 64 == k)[0]
        if rows.size == 0:
            assert k == 2 and not s.mins[:, k].any() and not s.scales[:, k].any()
            continue
        assert np.array_equal(rows, np.arange(rows[0], rows[-1] + 1))  # consecutive compact rows
        mn, mx = delta[rows].min(axis=0), delta[rows].max(axis=0)
        scale = ((mx - mn) / np.float32(15)).astype(np.float32)
        assert np.array_equal(s.mins[:, k, :], mn.astype(np.float16).view(np.uint16))
        assert np.array_equal(s.scales[:, k, :], scale.astype(np.float16).view(np.uint16))
        # every code is the nearest of the group's 16 FP32 levels
        lv = mn[None] + scale[None] * codes[rows]
        err = np.abs(delta[rows] - lv)
        assert np.all(err <= scale[None] / 2 * (1 + 1e-6) + 1e-30)


def test_tile_grouping_is_local_to_a_tile():
    """The point of tile grouping: changing the residual rows of one logical
    tile changes that tile's codes and K params only. Compact grouping offers
    no such bound (its groups straddle tiles)."""
    T, H, D = 300, 2, 128
    xs, a = _tile_chain(T, H, D, 22)
    x3 = f32(xs[2]).copy()
    hit = a[(a // 64) == 3]
    x3[hit] += 0.75
    xs_b = xs[:2] + [bf16(x3)]
    for kgroup in (O.KGROUP_TILE, O.KGROUP_COMPACT):
        s0 = O.encode_chain(O.KIND_K, xs[:3], [None, None, a], kgroup=kgroup)[2]
        s1 = O.encode_chain(O.KIND_K, xs_b, [None, None, a], kgroup=kgroup)[2]
        inside = (a // 64) == 3
        rows_changed = np.any(s0.codes != s1.codes, axis=(0, 2))
        groups_changed = np.any(s0.mins != s1.mins, axis=(0, 2)) | np.any(s0.scales != s1.scales, axis=(0, 2))
        if kgroup == O.KGROUP_TILE:
            assert not rows_changed[~inside].any()
            assert np.array_equal(np.nonzero(groups_changed)[0], [3])
        else:  # some row outside tile 3 shares a group with tile 3's rows and is re-coded
            assert rows_changed[~inside].any()


def test_tile_grouping_dense_bytes_and_chain_decode():
    """Dense loops group the same rows under both groupings (identical bytes);
    the sparse loop decodes through its tile's params: the FP32 chain step of a
    stored token t equals min16[t // 64] + scale16[t // 64] * code."""
    T, H, D = 200, 2, 128
    xs, a = _tile_chain(T, H, D, 23, drop_tile=1)
    acts = [None, None, a, a[::2].copy()]
    kt = O.encode_chain(O.KIND_K, xs, acts, kgroup=O.KGROUP_TILE)
    kc = O.encode_chain(O.KIND_K, xs, acts)
    for j in (0, 1):
        assert np.array_equal(kt[j].codes, kc[j].codes) and np.array_equal(kt[j].mins, kc[j].mins)
        assert np.array_equal(kt[j].scales, kc[j].scales)
    f2, f3 = O.decode_f32(kt, 2), O.decode_f32(kt, 3)
    s = kt[2]
    codes = unpack(s.codes)
    for i, t in enumerate(a):
        m = f16_to_f32(s.mins[:, t // 64, :])
        sc = f16_to_f32(s.scales[:, t // 64, :])
        step = (m + (sc * codes[i]).astype(np.float32)).astype(np.float32)
        assert np.array_equal(f3[t], (f2[t] + step).astype(np.float32))
    absent = np.setdiff1d(np.arange(T), a)
    assert np.array_equal(f3[absent], f2[absent])
    # the BF16 reconstruction agrees with the FP32 decode within its rounding
    rec = f32(O.reconstruct(kt, 4))
    assert np.max(np.abs(rec - O.decode_f32(kt, 4))) < 0.05


def test_tile_grouping_storage():
    """Tile grouping stores ceil(T/64) K groups per (head, channel) for a
    sparse loop, whatever its number of stored rows (an empty stream stores
    none); V and dense streams are unchanged."""
    H, D = 8, 128
    for n, T in ((130, 300), (1, 1000), (64, 64)):
        assert O.stream_bytes(O.KIND_K, n, H, D, sparse=True, T=T, kgroup=O.KGROUP_TILE) == \
            n * H * 64 + 2 * 2 * (-(-T // 64)) * H * D + 4 * n
        assert O.stream_bytes(O.KIND_V, n, H, D, sparse=True, T=T, kgroup=O.KGROUP_TILE) == \
            O.stream_bytes(O.KIND_V, n, H, D, sparse=True)
    assert O.stream_bytes(O.KIND_K, 0, H, D, sparse=True, T=300, kgroup=O.KGROUP_TILE) == 0
    assert O.stream_bytes(O.KIND_K, 300, H, D, sparse=False, T=300, kgroup=O.KGROUP_TILE) == \
        O.stream_bytes(O.KIND_K, 300, H, D)
    xs, a = _tile_chain(300, H, D, 24)
    s = O.encode_chain(O.KIND_K, xs[:3], [None, None, a], kgroup=O.KGROUP_TILE)[2]
    assert s.codes.nbytes + s.mins.nbytes + s.scales.nbytes + 4 * a.size == \
        O.stream_bytes(O.KIND_K, a.size, H, D, sparse=True, T=300, kgroup=O.KGROUP_TILE)


def test_rejects_unsorted_or_out_of_range_active():
    x = bf16(np.zeros((8, 1, 2), dtype=np.float32))
    for bad in ([3, 1], [1, 1], [-1, 2], [2, 8]):
        with pytest.raises(ValueError):
            O.encode(O.KIND_K, x, x, np.array(bad, dtype=np.int32))


# ---------------------------------------------------------------- storage accounting


def test_storage_sizes_closed_form():
    gold = json.load(open(os.path.join(GOLD, "storage.json")))
    H, D = 8, 128
    for n in (64, 128, 4096):  # full groups: 4 bits of code + 32 bits of params per 64 elements
        for kind in (O.KIND_K, O.KIND_V):
            bits = O.stream_bytes(kind, n, H, D) * 8 / (n * H * D)
            assert bits == gold["bits_per_element_full_groups"]
    # partial groups pay their padding: ceil(n/64) K groups
    assert O.stream_bytes(O.KIND_K, 65, H, D) == 65 * H * 64 + 2 * 2 * 2 * H * D
    assert O.stream_bytes(O.KIND_V, 65, H, D) == 65 * H * 64 + 2 * 2 * 65 * H * 2
    assert O.stream_bytes(O.KIND_K, 65, H, D, sparse=True) == O.stream_bytes(O.KIND_K, 65, H, D) + 4 * 65
    # the stored byte arrays have exactly these sizes
    x = bf16(np.random.default_rng(0).standard_normal((65, H, D)))
    for kind in (O.KIND_K, O.KIND_V):
        s = O.encode(kind, x)
        assert s.codes.nbytes + s.mins.nbytes + s.scales.nbytes == O.stream_bytes(kind, 65, H, D)
    # payload-only ratio of four BF16 depths vs INT4 at retention [1, 1, 0.25, 0.10]
    N = 6400
    code_bytes = sum(O.encode(O.KIND_V, bf16(np.zeros((int(r * N), 1, 2), np.float32))).codes.nbytes
                     for r in gold["retention"])
    ratio = (4 * N * 16) / (code_bytes * 8 / 2)  # one code byte holds two channels
    assert abs(ratio - 64 / 9.4) < 1e-9
    assert round(ratio, 2) == gold["payload_ratio_about"]


# ---------------------------------------------------------------- decode attention


def _sdpa64(q, k, v, scale):
    """Float64 reference through torch's scaled_dot_product_attention (GQA)."""
    Hq, D = q.shape
    T, H, _ = k.shape
    g = Hq // H
    qt = torch.from_numpy(f32(q).astype(np.float64)).reshape(1, Hq, 1, D)
    kt = torch.from_numpy(f32(k).astype(np.float64)).permute(1, 0, 2).repeat_interleave(g, 0).unsqueeze(0)
    vt = torch.from_numpy(f32(v).astype(np.float64)).permute(1, 0, 2).repeat_interleave(g, 0).unsqueeze(0)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o.reshape(Hq, D).numpy()


@pytest.mark.parametrize("T,H,Hq", [(1, 2, 8), (7, 2, 8), (300, 8, 32), (513, 8, 64), (100, 4, 4)])
def test_attention_matches_float64_sdpa(T, H, Hq):
    rng = np.random.default_rng(T + Hq)
    D = 128
    q = bf16(rng.standard_normal((Hq, D)))
    k = bf16(rng.standard_normal((T, H, D)) * 1.5)
    v = bf16(rng.standard_normal((T, H, D)))
    scale = 1.0 / math.sqrt(D)
    out = O.attention(q, k, v, scale)
    ref = _sdpa64(q, k, v, scale)
    assert np.max(np.abs(out - ref)) < 2e-5


def test_attention_special_cases():
    rng = np.random.default_rng(5)
    D, H, Hq = 128, 2, 8
    v1 = bf16(rng.standard_normal((1, H, D)))
    out = O.attention(bf16(rng.standard_normal((Hq, D))), bf16(rng.standard_normal((1, H, D))), v1, 0.088)
    for hq in range(Hq):  # one stored token: the output is that token's value
        assert np.array_equal(out[hq], f32(v1)[0, hq // 4])
    T = 37
    v = bf16(rng.standard_normal((T, H, D)))
    out = O.attention(bf16(np.zeros((Hq, D))), bf16(rng.standard_normal((T, H, D))), v, 0.088)
    mean = f32(v).astype(np.float64).mean(axis=0)  # equal logits: the plain mean
    for hq in range(Hq):
        assert np.max(np.abs(out[hq] - mean[hq // 4])) < 1e-6


# ---------------------------------------------------------------- FP32 decode of the packed chain


def test_decode_f32_depth1_is_the_affine_decode():
    """FlashLoop RFC §3.3: decoding is min + scale * code. At depth 1 the FP32
    decode is that value rounded once to FP32, and its BF16 rounding is the
    BF16 reconstruction bit for bit."""
    rng = np.random.default_rng(21)
    x = bf16(rng.standard_normal((70, 2, 128)) * 3)
    for kind in (O.KIND_K, O.KIND_V):
        s = O.encode(kind, x)
        f = O.decode_f32([s], 1)
        assert np.array_equal(O.f32_to_bf16_bits(f), O.reconstruct([s], 1))
        c = unpack(s.codes)
        for (t, h, d) in [(0, 0, 0), (5, 1, 77), (69, 0, 127), (64, 1, 63), (33, 0, 64)]:
            p = (h, t // 64, d) if kind == O.KIND_K else (h, t, d // 64)
            exact = Fraction(float(f16_to_f32(s.mins[p]))) + Fraction(float(f16_to_f32(s.scales[p]))) * int(c[t, h, d])
            assert float(f[t, h, d]) == float(np.float32(float(exact)))


def test_decode_f32_inherits_absent_tokens_and_tracks_the_bf16_chain():
    gold = json.load(open(os.path.join(GOLD, "loop4_read_example.json")))
    act = {int(r): np.array(v, dtype=np.int32) - 1 for r, v in gold["active_1based"].items()}
    xs = _offset_chain(gold["T"], 2, 128, 6)
    for kind in (O.KIND_K, O.KIND_V):
        ks = O.encode_chain(kind, xs, [None, None, act[3], act[4]])
        f = {d: O.decode_f32(ks, d) for d in range(1, 5)}
        for tok1, loops in gold["loop4_read_1based"].items():
            t = int(tok1) - 1
            for d in range(2, 5):
                assert (not np.array_equal(f[d][t], f[d - 1][t])) == (d in loops)
        # the FP32 chain and the BF16 chain differ only by the 2*depth-1 BF16 roundings
        for d in range(1, 5):
            bf = f32(O.reconstruct(ks, d)).astype(np.float64)
            mag = np.maximum(np.abs(bf), np.abs(f[d].astype(np.float64)))
            assert np.all(np.abs(bf - f[d]) <= (2 * d - 1) * 2.0 ** -8 * (mag + 4.0))


def test_attention_f32_matches_float64_sdpa_on_decoded_chain():
    rng = np.random.default_rng(4)
    T, H, Hq, D = 333, 4, 16, 128
    xs = [bf16(rng.standard_normal((T, H, D)) * (0.1 if r else 1.0)) for r in range(4)]
    xs = [bf16(sum(f32(xs[i]) for i in range(r + 1))) for r in range(4)]
    ks = O.encode_chain(O.KIND_K, xs, [None] * 4)
    vs = O.encode_chain(O.KIND_V, xs, [None] * 4)
    kf, vf = O.decode_f32(ks, 4), O.decode_f32(vs, 4)
    q = bf16(rng.standard_normal((Hq, D)))
    out = O.attention_f32(q, kf, vf, 1 / math.sqrt(D))
    g = Hq // H
    qt = torch.from_numpy(f32(q).astype(np.float64)).reshape(1, Hq, 1, D)
    kt = torch.from_numpy(kf.astype(np.float64)).permute(1, 0, 2).repeat_interleave(g, 0).unsqueeze(0)
    vt = torch.from_numpy(vf.astype(np.float64)).permute(1, 0, 2).repeat_interleave(g, 0).unsqueeze(0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=1 / math.sqrt(D)).reshape(Hq, D)
    assert np.max(np.abs(out - ref.numpy())) < 2e-5



# ---------------------------------------------------------------- direct-reader error bound


def _nested_chain(T, H, D, seed, sparse):
    rng = np.random.default_rng(seed)
    xs = [rng.standard_normal((T, H, D)).astype(np.float32) * 2.0]
    for r in range(1, 4):
        xs.append(xs[-1] + 0.1 * rng.standard_normal((T, H, D)).astype(np.float32))
    acts = [None, None, None, None]
    if sparse:
        a3 = np.sort(rng.choice(T, size=(T + 1) // 2, replace=False)).astype(np.int32)
        a4 = np.sort(rng.choice(a3, size=(len(a3) + 1) // 2, replace=False)).astype(np.int32)
        acts = [None, None, a3, a4]
    return [bf16(x) for x in xs], acts


@pytest.mark.parametrize("sparse", [False, True])
def test_chain_gap_recurrence_bounds_bf16_vs_fp32_chain(sparse):
    """The per-element gap between the BF16 reconstruction and the FP32 decode
    stays within the rounding recurrence of tests/reader_bound.py at every
    depth, and the recurrence is tight (within 2x of the largest gap). A chain
    read one loop short on the FP32 side breaks it."""
    xs, acts = _nested_chain(150, 2, 128, 31 + sparse, sparse)
    for kind in (O.KIND_K, O.KIND_V):
        st = O.encode_chain(kind, xs, acts)
        for d in range(1, 5):
            b = RB.chain_gap_bound(st, d)
            gap = np.abs(f32(O.reconstruct(st, d)).astype(np.float64) - O.decode_f32(st, d))
            assert np.all(gap <= b)
            assert (gap / np.maximum(b, 1e-300)).max() > 0.5
        short = np.abs(f32(O.reconstruct(st, 4)).astype(np.float64) - O.decode_f32(st, 3))
        assert np.any(short > RB.chain_gap_bound(st, 4))


def test_softmax_shift_bound_holds_for_large_shifts():
    """The second-order bound on a softmax-weighted sum under score and value
    shifts, checked against the exact float64 value for shifts up to 0.5."""
    rng = np.random.default_rng(9)
    for trial in range(200):
        T, D = int(rng.integers(1, 300)), 8
        s = rng.standard_normal(T) * float(rng.choice([0.1, 1.0, 5.0]))
        e = rng.standard_normal(T) * float(rng.choice([1e-4, 1e-2, 0.1, 0.25]))
        vf = rng.standard_normal((T, D))
        vh = vf + rng.standard_normal((T, D)) * 1e-3
        w0 = np.exp(s - s.max())
        w0 /= w0.sum()
        w1 = np.exp(s + e - (s + e).max())
        w1 /= w1.sum()
        exact = np.abs(w1 @ vh - w0 @ vf)
        b = RB.softmax_shift_bound(s, e, vh, vf)
        assert np.all(exact <= b), trial
        if np.abs(e).max() <= 1e-2:  # small shifts: the bound is essentially the exact value
            assert b.max() <= 1.1 * exact.max() + 1e-6, trial


@pytest.mark.parametrize("sparse,depth", [(False, 1), (False, 4), (True, 3), (True, 4)])
def test_reader_error_bound_holds(sparse, depth):
    """FlashLoop RFC §9: the attention over the BF16 reconstruction and the FP32
    attention over the FP32 decode differ by at most the derived bound; a V
    chain read one loop short exceeds it."""
    xk, acts = _nested_chain(300, 2, 128, 41 + depth, sparse)
    xv, _ = _nested_chain(300, 2, 128, 51 + depth, sparse)
    ks = O.encode_chain(O.KIND_K, xk, acts)
    vs = O.encode_chain(O.KIND_V, xv, acts)
    q = bf16(np.random.default_rng(3).standard_normal((8, 128)))
    scale = 1 / math.sqrt(128)
    o_f32 = O.attention_f32(q, O.decode_f32(ks, depth), O.decode_f32(vs, depth), scale).astype(np.float64)
    o_bf = O.attention(q, O.reconstruct(ks, depth), O.reconstruct(vs, depth), scale).astype(np.float64)
    b = RB.reader_error_bound(q, ks, vs, depth, scale)
    assert np.all(np.abs(o_bf - o_f32) <= b)
    assert b.max() < 2e-2
    if depth > 1:
        o_short = O.attention(q, O.reconstruct(ks, depth), O.reconstruct(vs, depth - 1), scale).astype(np.float64)
        assert np.any(np.abs(o_short - o_f32) > b)


# ---------------------------------------------------------------- BF16 sink and tail segments


def _sdpa64_rows(q, krows, vrows, scale, Hq):
    """float64 SDPA over explicit K/V rows [N, H, D] (float64 arrays)."""
    N, H, D = krows.shape
    g = Hq // H
    qt = torch.from_numpy(f32(q).astype(np.float64)).reshape(1, Hq, 1, D)
    kt = torch.from_numpy(krows).permute(1, 0, 2).repeat_interleave(g, 0).unsqueeze(0)
    vt = torch.from_numpy(vrows).permute(1, 0, 2).repeat_interleave(g, 0).unsqueeze(0)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale).reshape(Hq, D).numpy()


def test_segments_absent_is_the_chain_attention():
    rng = np.random.default_rng(31)
    T, H, Hq, D = 90, 2, 8, 128
    kf = rng.standard_normal((T, H, D)).astype(np.float32)
    vf = rng.standard_normal((T, H, D)).astype(np.float32)
    q = bf16(rng.standard_normal((Hq, D)))
    empty = np.zeros((0, H, D), dtype=np.uint16)
    a = O.attention_f32(q, kf, vf, 0.088)
    assert np.array_equal(O.attention_with_segments(q, kf, vf, 0.088), a)
    assert np.array_equal(O.attention_with_segments(q, kf, vf, 0.088, empty, empty, empty, empty), a)


@pytest.mark.parametrize("T,ns,nt", [(90, 4, 64), (64, 64, 127), (0, 0, 100), (130, 0, 1), (70, 3, 0)])
def test_segments_replace_the_sink_and_append_the_tail(T, ns, nt):
    """FlashLoop RFC §3.3 rolling BF16 tail and the BF16 sink of the codec PR
    review: against float64 attention over the rows assembled independently
    (sink values for the first tokens, chain values after them, tail last)."""
    rng = np.random.default_rng(T + 7 * ns + nt)
    H, Hq, D = 2, 8, 128
    kf = rng.standard_normal((T, H, D)).astype(np.float32)
    vf = rng.standard_normal((T, H, D)).astype(np.float32)
    sk, sv = bf16(rng.standard_normal((ns, H, D))), bf16(rng.standard_normal((ns, H, D)))
    tk, tv = bf16(rng.standard_normal((nt, H, D))), bf16(rng.standard_normal((nt, H, D)))
    q = bf16(rng.standard_normal((Hq, D)))
    out = O.attention_with_segments(q, kf, vf, 0.088, sk, sv, tk, tv)
    krows = np.concatenate([f32(sk).astype(np.float64), kf[ns:].astype(np.float64), f32(tk).astype(np.float64)])
    vrows = np.concatenate([f32(sv).astype(np.float64), vf[ns:].astype(np.float64), f32(tv).astype(np.float64)])
    assert krows.shape[0] == T + nt
    ref = _sdpa64_rows(q, krows, vrows, 0.088, Hq)
    assert np.max(np.abs(out - ref)) < 2e-5
    # the sink replaces tokens: the original chain values of those tokens are not read
    if ns:
        kf2, vf2 = kf.copy(), vf.copy()
        kf2[:ns] += 100.0
        vf2[:ns] -= 50.0
        assert np.array_equal(O.attention_with_segments(q, kf2, vf2, 0.088, sk, sv, tk, tv), out)


def test_segments_nothing_to_attend_is_zero():
    q = bf16(np.ones((8, 128)))
    z = np.zeros((0, 2, 128), dtype=np.float32)
    assert np.array_equal(O.attention_with_segments(q, z, z, 0.1), np.zeros((8, 128), dtype=np.float32))


# ---------------------------------------------------------------- sparse decode attention


def test_sparse_scalar_example():
    """The RFC §3.2 worked example, with one channel and logits log(p)."""
    gold = json.load(open(os.path.join(GOLD, "sparse_scalar_example.json")))
    one = bf16(np.ones((1, 1)))
    kr = np.log(np.array(gold["ref_probs"]))[:, None, None]
    vr = np.array(gold["ref_values"])[:, None, None]
    S, m, o_ref, c_ref = O.sparse_reference(one, kr, vr, 1.0, gold["n_select"])
    assert S[0].tolist() == gold["selected"]
    assert abs(m[0] - gold["mass"]) < 1e-12
    assert abs(o_ref[0, 0] - gold["o_ref"]) < 1e-12
    assert abs(c_ref[0, 0] - gold["c_ref"]) < 1e-12
    k_new = np.zeros((3, 1, 1))
    v_new = np.zeros((3, 1, 1))
    k_new[S[0], 0, 0] = np.log(np.array(gold["later_probs_on_selected"]))
    v_new[S[0], 0, 0] = gold["later_values_on_selected"]
    k_new[0, 0, 0] = 50.0  # an unselected key: not read at the later loop
    out = O.sparse_decode(one, k_new, v_new, 1.0, S, m, o_ref, c_ref)
    assert abs(out[0, 0] - gold["o_new"]) < 1e-12


def test_sparse_all_keys_is_dense_attention():
    """With every key retained, m = 1 and C_ref = O_ref, so the later loop is
    plain dense attention over its own keys (RFC §3.2)."""
    rng = np.random.default_rng(12)
    T, H, Hq, D = 50, 2, 8, 128
    q = bf16(rng.standard_normal((Hq, D)))
    k0, v0 = rng.standard_normal((T, H, D)), rng.standard_normal((T, H, D))
    k1, v1 = rng.standard_normal((T, H, D)), rng.standard_normal((T, H, D))
    S, m, o_ref, c_ref = O.sparse_reference(q, k0, v0, 0.09, T)
    assert np.allclose(m, 1.0) and np.allclose(c_ref, o_ref)
    out = O.sparse_decode(q, k1, v1, 0.09, S, m, o_ref, c_ref)
    assert np.max(np.abs(out - _sdpa64_rows(q, k1, v1, 0.09, Hq))) < 1e-9


def test_sparse_later_loop_on_the_reference_keys_returns_o_ref():
    """A later loop that reads the reference loop's own K and V with the same
    query attends S with the probabilities p_t / m, so m * softmax_S(V) = C_ref
    and O = O_ref - C_ref + C_ref = O_ref, whatever the budget (RFC §3.2). A
    dropped correction term, a wrong sign or a mass not taken over S breaks it."""
    rng = np.random.default_rng(14)
    T, H, Hq, D = 37, 2, 8, 128
    q = bf16(rng.standard_normal((Hq, D)))
    k, v = rng.standard_normal((T, H, D)), rng.standard_normal((T, H, D))
    for K in (1, 5, 20, 36):
        S, m, o_ref, c_ref = O.sparse_reference(q, k, v, 0.09, K)
        assert np.all((m > 0) & (m < 1))
        out = O.sparse_decode(q, k, v, 0.09, S, m, o_ref, c_ref)
        assert np.max(np.abs(out - o_ref)) < 1e-9, K
        # and the output moves when the later loop's values do
        out2 = O.sparse_decode(q, k, v + 1.0, 0.09, S, m, o_ref, c_ref)
        assert np.allclose(out2 - o_ref, m[:, None]), K


def test_sparse_selection_is_top_k_with_position_ties():
    rng = np.random.default_rng(13)
    T, H, Hq, D = 40, 1, 2, 128
    q = bf16(rng.standard_normal((Hq, D)))
    k = rng.standard_normal((T, H, D))
    k[10] = k[30] = k[5]  # three equal logits
    for K in (1, 7, 20, 40, 55):
        S, m, _, _ = O.sparse_reference(q, k, k, 0.1, K)
        assert S.shape == (Hq, min(K, T))
        for hq in range(Hq):
            s = k[:, 0, :] @ f32(q)[hq].astype(np.float64) * 0.1
            brute = sorted(range(T), key=lambda t: (-s[t], t))[:min(K, T)]
            assert S[hq].tolist() == sorted(brute)
            p = np.exp(s - s.max())
            assert abs(m[hq] - p[sorted(brute)].sum() / p.sum()) < 1e-12


# ---------------------------------------------------------------- NVFP4 residual (codec PR review by 0z5a)


def test_e4m3_matches_torch_float8_cast():
    """E4M3 rounding (round to nearest even) agrees with torch's float8_e4m3fn cast
    (a library routine) below its overflow point; above 448 the oracle saturates."""
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.uniform(0, 464, 200_000), np.exp(rng.uniform(np.log(1e-6), np.log(464), 200_000)),
        np.arange(0, 4096) / 4096 * 2 ** -6,                # subnormal range and its ties
        (np.arange(1, 2048) / 8.0 + 0.0625) * 2.0 ** rng.integers(-6, 8, 2047),  # mantissa ties
    ]).astype(np.float32)
    x = x[x < 464]
    for sign in (1, -1):
        got = O.f32_to_e4m3_bits(sign * x)
        ref = torch.from_numpy(sign * x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(got, ref)
    assert np.all(O.f32_to_e4m3_bits(np.array([464.0, 500.0, 1e30], np.float32)) == 0x7E)
    # decoding every finite pattern agrees with torch's float8 view
    bits = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    assert np.array_equal(O.e4m3_bits_to_f32(bits), ref)


def test_e2m1_is_nearest_with_ties_to_even():
    """E2M1 codes: the nearest of the eight magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6
    (exact rational distances), ties to the even code, above 6 saturating; the
    sign bit follows the input's sign."""
    mags = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4),
            Fraction(6)]
    assert list(O.e2m1_bits_to_f32(np.arange(8))) == [float(m) for m in mags]
    assert list(O.e2m1_bits_to_f32(np.arange(8, 16))) == [-float(m) for m in mags]
    vals = np.concatenate([np.arange(0, 8.5, 1 / 64), np.random.default_rng(6).uniform(0, 7, 5000)]).astype(np.float32)
    for sign in (1.0, -1.0):
        codes = O.f32_to_e2m1_bits(sign * vals)
        for v, c in zip(vals, codes):
            fv = Fraction(float(v))
            if fv > 6:
                assert c & 7 == 7
            else:
                d = [abs(fv - m) for m in mags]
                best = min(d)
                cands = [k for k in range(8) if d[k] == best]
                want = cands[0] if len(cands) == 1 else [k for k in cands if k % 2 == 0][0]
                assert c & 7 == want, (float(v), c)
            assert (c >> 3) == (1 if sign < 0 else 0)


def _nvfp4_case(T, H, D, seed, sparse):
    xs = _offset_chain(T, H, D, seed)
    act = None
    if sparse:
        act = np.sort(np.random.default_rng(seed).choice(T, T // 2, replace=False)).astype(np.int32)
    base = O.encode(O.KIND_K, xs[0])
    pred = O.reconstruct([base], 1)
    s = O.encode_nvfp4(O.KIND_K, xs[1], pred, act)
    rows = act if act is not None else np.arange(T)
    delta = f32(bf16(f32(xs[1])[rows] - f32(pred)[rows]))  # [n, H, D] compact order
    return s, delta


@pytest.mark.parametrize("sparse", [False, True])
def test_nvfp4_scales_follow_the_two_level_recipe(sparse):
    """Codec PR review by 0z5a (NVFP4: E2M1 elements, one E4M3 scale per 16
    elements, one FP32 scale per tensor): s_t = amax/(6·448) in FP32; each
    block of 16 channels of one (row, head) stores E4M3(a_b / (6 s_t)) (torch's
    float8 cast), and the block holding the tensor's largest |δ| gets 448."""
    T, H, D = 130, 4, 128
    s, delta = _nvfp4_case(T, H, D, 31, sparse)
    amax = np.float32(np.abs(delta).max())
    st = np.float32(amax / np.float32(2688))
    assert s.tscale[0] == st
    blk = np.abs(delta).reshape(delta.shape[0], H, D // 16, 16).max(axis=3)  # [n, H, D/16]
    want = torch.from_numpy((blk / np.float32(np.float32(6) * st)).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(np.transpose(s.bscale, (1, 0, 2)), want)
    where = np.unravel_index(np.argmax(np.abs(delta)), delta.shape)
    assert O.e4m3_bits_to_f32(s.bscale[where[1], where[0], where[2] // 16]) == 448.0


@pytest.mark.parametrize("sparse", [False, True])
def test_nvfp4_codes_are_nearest_levels(sparse):
    """Each code is the E2M1 value nearest to δ / (s_b · s_t) with the sign of δ;
    the decode error is at most one quantisation step e_b = s_b · s_t."""
    T, H, D = 70, 2, 128
    s, delta = _nvfp4_case(T, H, D, 32, sparse)
    n = delta.shape[0]
    codes = unpack(s.codes)  # [n, H, D]
    sb = O.e4m3_bits_to_f32(np.transpose(s.bscale, (1, 0, 2)))  # [n, H, D/16]
    eb = (np.repeat(sb, 16, axis=2) * s.tscale[0]).astype(np.float32)
    vals = O.e2m1_bits_to_f32(codes)
    y = (delta / eb).astype(np.float32)  # IEEE FP32 division, like the quantiser
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    dist = np.abs(np.abs(y)[..., None] - mags)
    best = dist.min(axis=-1)
    assert np.all(np.abs(np.abs(y) - np.abs(vals)) == best)  # a nearest magnitude (ties checked below)
    neg = np.signbit(y)
    assert np.array_equal(codes >= 8, neg)
    tie = (dist == best[..., None]).sum(axis=-1) > 1
    assert np.all((codes[tie] & 7) % 2 == 0)
    dq = (vals * np.repeat(sb, 16, axis=2)).astype(np.float32) * s.tscale[0]
    assert np.all(np.abs(delta - dq) <= eb * 1.0001)
    assert n == (T // 2 if sparse else T)


def test_nvfp4_zero_stream_and_chain_decode():
    """A residual that vanishes stores s_t = 0 and zero codes; the chain decodes
    an NVFP4 loop as e2m1 · s_b · s_t at its stored rows (absent rows inherit),
    and the BF16 reconstruction rounds that step to BF16 before the add."""
    T, H, D = 100, 2, 128
    xs = _offset_chain(T, H, D, 33)
    base = O.encode(O.KIND_V, xs[0])
    pred = O.reconstruct([base], 1)
    z = O.encode_nvfp4(O.KIND_V, pred, pred)  # X_2 = X̂_1: δ = 0 everywhere
    assert z.tscale[0] == 0 and not z.codes.any() and not z.bscale.any()
    assert np.array_equal(O.reconstruct([base, z], 2), pred)
    act = np.sort(np.random.default_rng(3).choice(T, 37, replace=False)).astype(np.int32)
    ch = O.encode_chain(O.KIND_K, xs, [None, None, act, act[::3].copy()],
                        formats=[O.FMT_INT4, O.FMT_NVFP4, O.FMT_NVFP4, O.FMT_NVFP4])
    f2, f3 = O.decode_f32(ch, 2), O.decode_f32(ch, 3)
    s = ch[2]
    codes = unpack(s.codes)
    sb = O.e4m3_bits_to_f32(np.transpose(s.bscale, (1, 0, 2)))
    step = (O.e2m1_bits_to_f32(codes) * np.repeat(sb, 16, axis=2)).astype(np.float32) * s.tscale[0]
    assert np.array_equal(f3[act], (f2[act] + step).astype(np.float32))
    absent = np.setdiff1d(np.arange(T), act)
    assert np.array_equal(f3[absent], f2[absent])
    r2, r3 = f32(O.reconstruct(ch, 2)), f32(O.reconstruct(ch, 3))
    assert np.array_equal(r3[act], f32(bf16(r2[act] + f32(bf16(step)))))
    assert np.max(np.abs(f32(O.reconstruct(ch, 4)) - O.decode_f32(ch, 4))) < 0.05


def test_nvfp4_storage():
    """4 bits of code and one E4M3 byte per 16 elements: 4.5 bits per element,
    plus the 4-byte tensor scale (codec PR review by 0z5a: NVFP4 ties INT4's
    4.5 bits)."""
    H, D = 8, 128
    for n in (64, 1000, 4096):
        bits = O.stream_bytes_nvfp4(n, H, D) * 8 / (n * H * D)
        assert abs(bits - (4.5 + 32 / (n * H * D))) < 1e-12
        assert O.stream_bytes_nvfp4(n, H, D, sparse=True) == O.stream_bytes_nvfp4(n, H, D) + 4 * n
    assert O.stream_bytes_nvfp4(0, H, D) == 0
    s, _ = _nvfp4_case(130, H, D, 34, False)
    assert s.codes.nbytes + s.bscale.nbytes + s.tscale.nbytes == O.stream_bytes_nvfp4(130, H, D)
