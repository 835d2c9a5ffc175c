"""The direct-reader error, derived from the rounding steps of the chain.

FlashLoop RFC §9 (algorithm and runtime correctness, KV) asks the packed
direct reader's error to be bounded. Two attentions are compared:

- the reference of the direct reader: FP32 attention over X̃, the FP32 decode
  of the packed chain (decode = RN32(min + RN32(scale * code)), loops summed in
  FP32, no BF16 rounding);
- the attention over X̂, the BF16 reconstruction of the chain (RFC §3.3, codec
  PR "subtraction/addition in the input compute dtype"): every decoded value
  is rounded to BF16 and every chain add rounds to BF16.

Chain gap (per element). Let u = 2^-8 (BF16: 8 significant bits, round to
nearest) and v = 2^-24 (FP32). With dec_j the FP32 decode of loop j:
    X̂_1 = RN_bf16(dec_1),        X̃_1 = dec_1
    X̂_j = RN_bf16(RN32(S_j)),    S_j = X̂_{j-1} + RN_bf16(dec_j)
    X̃_j = RN32(X̃_{j-1} + dec_j)
so e_j = X̂_j - X̃_j obeys
    |e_1| <= u |X̃_1|
    |e_j| <= |e_{j-1}| + u |dec_j| + w |S_j| + v |X̃_j| / (1 - v)   (token stored in loop j)
    |e_j| =  |e_{j-1}|                                               (token absent: both inherit)
with w = v + u (1 + v) the relative error of RN_bf16(RN32(.)), |S_j| <= |X̂_j| /
(1 - w) and |dec_j| <= |X̃_j - X̃_{j-1}| + v |X̃_j|.

Attention. For one query head (kv head h), let w_t = softmax(s~)_t be the
weights over X~ and e_t = s^_t - s~_t = scale * q . (k^_t - k~_t) the score
shift (computed from the packed data: both decodes of the same chain). With
x_t = e_t - sum_u w_u e_u, the weights over X^ are w_t exp(x_t) / Z, Z = sum_u
w_u exp(x_u). Writing exp(x) = 1 + x + r(x), |r(x)| <= x^2 exp(|x|) / 2, and
c_d = sum_t w_t v^_td, P = sum_t w_t r(x_t):
    sum_t (w^_t - w_t) v^_td = (A_d + B_d) / (1 + P),
    A_d = sum_t w_t x_t (v^_td - c_d),   |B_d| <= X^2 exp(X) / 2 * sum_t w_t |v^_td - c_d|,
where X = max_t |x_t| and |P| <= X^2 exp(X) / 2. Since
o(X^) - o(X~) = sum_t (w^_t - w_t) v^_td + sum_t w_t (v^_td - v~_td),
    |o(X^) - o(X~)|_d <= |A_d + sum_t w_t dV_td| + (|A_d| |P| + |B_d|) / (1 - |P|).
The first-order part is evaluated from the actual gaps (their signs matter: a
bound from |q| . gapK alone, with no sign information, is about 1.5 on these
inputs, far above the 2e-3 attention tolerance); the remainder is rigorous.
The per-element gaps themselves are held to the recurrence above.

Evaluation of the two FP32 oracle attentions. Each computes s_t as an FP32
dot product in channel order (error <= g_{D+1} scale sum_d |q_d k_td|, with
g_n = n v / (1 - n v)), exp of s_t - max (a few ulp), and FP32 sums over t
(error <= g_T of the sum of magnitudes). Its distance to the exact attention
over the same values is at most (exp(2 E_e) - 1) R_d / 2 + (2 g_T + 2 v) max_t
|v_td| with E_e = g_{D+2} scale max_t sum_d |q_d k_td| + 4 v (1 + 2 max_t |s_t|).
"""

from __future__ import annotations

import numpy as np

from oracle import oracle as O

U_BF16 = 2.0 ** -8
U_F32 = 2.0 ** -24
W_BF16_F32 = U_F32 + U_BF16 * (1.0 + U_F32)


def _g(n: int) -> float:
    return n * U_F32 / (1.0 - n * U_F32)


def _present(stream, T: int) -> np.ndarray:
    if stream.active is None:
        return np.ones(T, dtype=bool)
    m = np.zeros(T, dtype=bool)
    m[np.asarray(stream.active, dtype=np.int64)] = True
    return m


def chain_gap_bound(streams, depth: int) -> np.ndarray:
    """float64 [T, H, D]: an upper bound on |X̂ - X̃| per element at `depth`,
    following the recurrence in the module docstring."""
    T = streams[0].T
    xt_prev = O.decode_f32(streams, 1).astype(np.float64)
    b = U_BF16 * np.abs(xt_prev)
    for j in range(2, depth + 1):
        xt = O.decode_f32(streams, j).astype(np.float64)
        xh = O.bf16_bits_to_f32(O.reconstruct(streams, j)).astype(np.float64)
        dec = np.abs(xt - xt_prev) + U_F32 * np.abs(xt)
        step = U_BF16 * dec + W_BF16_F32 * np.abs(xh) / (1.0 - W_BF16_F32) + U_F32 * np.abs(xt) / (1.0 - U_F32)
        b = b + np.where(_present(streams[j - 1], T)[:, None, None], step, 0.0)
        xt_prev = xt
    return b


def _eval_bound(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> float:
    """Distance of an FP32 oracle attention (one query head) to the exact one
    over the same K, V [T, D] (float64 arrays), per the docstring."""
    T, D = k.shape
    if T == 0:
        return 0.0
    mag = scale * (np.abs(k) @ np.abs(q))
    s = scale * (k @ q)
    e = _g(D + 2) * float(mag.max()) + 4.0 * U_F32 * (1.0 + 2.0 * float(np.abs(s).max()))
    r = v.max(axis=0) - v.min(axis=0)
    return np.expm1(2.0 * e) * r / 2.0 + (2.0 * _g(T) + 2.0 * U_F32) * np.abs(v).max(axis=0)


def softmax_shift_bound(s: np.ndarray, e: np.ndarray, vh: np.ndarray, vf: np.ndarray) -> np.ndarray:
    """Bound on |sum_t softmax(s + e)_t vh_t - sum_t softmax(s)_t vf_t| per
    channel (s, e: scores and score shifts [T]; vh, vf: values [T, D]), by the
    second-order expansion of the module docstring, in float64."""
    w = np.exp(s - s.max())
    w /= w.sum()
    x = e - w @ e
    X = float(np.abs(x).max())
    rmax = X * X * np.exp(X) / 2.0
    if rmax >= 1.0:
        return np.full(vh.shape[1], np.inf)
    dev = vh - w @ vh
    A = (w * x) @ dev
    Bm = rmax * (w @ np.abs(dev))
    first = np.abs(A + w @ (vh - vf))
    return first + (np.abs(A) * rmax + Bm) / (1.0 - rmax) + 1e-12 * (1.0 + np.abs(vh).max(axis=0))


def reader_error_bound(q_bits: np.ndarray, ks, vs, depth: int, scale: float) -> np.ndarray:
    """float64 [Hq, D]: a bound on |attention over X^ - attention over X~| per
    output element (second-order expansion around the actual chain gaps, see
    the module docstring), including the FP32 evaluation error of both oracle
    attentions (q_bits: BF16 bits [Hq, D])."""
    q = O.bf16_bits_to_f32(np.asarray(q_bits, dtype=np.uint16)).astype(np.float64)
    Hq, D = q.shape
    T, H = ks[0].T, ks[0].H
    out = np.zeros((Hq, D))
    if T == 0:
        return out
    g = Hq // H
    kf = O.decode_f32(ks, depth).astype(np.float64)
    vf = O.decode_f32(vs, depth).astype(np.float64)
    kh = O.bf16_bits_to_f32(O.reconstruct(ks, depth)).astype(np.float64)
    vh = O.bf16_bits_to_f32(O.reconstruct(vs, depth)).astype(np.float64)
    for hq in range(Hq):
        h = hq // g
        s = scale * (kf[:, h, :] @ q[hq])
        e = scale * ((kh[:, h, :] - kf[:, h, :]) @ q[hq])
        out[hq] = (softmax_shift_bound(s, e, vh[:, h, :], vf[:, h, :])
                   + _eval_bound(q[hq], kh[:, h, :], vh[:, h, :], scale)
                   + _eval_bound(q[hq], kf[:, h, :], vf[:, h, :], scale))
    return out
