"""Seeded synthetic inputs for the packed-KV path.

This module draws random numbers and nothing else: it holds none of the
codec, reconstruction or attention arithmetic, so the CPU oracle and the CUDA
path can both be fed from it.

Shapes follow the five synthetic configurations of the packed-KV hot path:
per request and layer, K and V for four recurrent loops as BF16 ``[T, H, D]``;
X1 ~ N(0, 1) and X_r = X_{r-1} + sigma * N(0, 1) accumulated in FP32, each
loop rounded to BF16 on its own; K and V from independent draws; one decode
query per request, ``q ~ N(0, 1)`` in BF16 ``[Hq, D]``. Loops 1 and 2 are
dense; a sparse loop keeps a sorted random subset whose size is
``ceil(ratio * T)`` of the original window and which is nested in the
previous sparse loop's set (FlashLoop RFC, vllm-rlt issue #156, §3.1:
budgets refer to the original window, active sets are nested).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class ConfigSpec:
    name: str
    seed: int
    n_requests: int
    T: int | None  # fixed length, or None for drawn lengths
    H: int
    D: int
    Hq: int
    loops: int
    sigma: float
    ratios: tuple  # per loop: 1.0 dense, else the sparse retention ratio
    k_outlier_frac: float = 0.0
    k_outlier_gain: float = 1.0
    ragged: tuple | None = None  # (lo, hi) for drawn lengths that avoid multiples of 64
    mixed: bool = False  # per request fair coin: dense or sparse late loops
    layers: int = 1


CONFIGS = {
    1: ConfigSpec("tiny", 0, 1, 256, 8, 128, 32, 4, 0.1, (1.0, 1.0, 1.0, 1.0)),
    2: ConfigSpec("partial_sparse", 1, 1, 1000, 8, 128, 32, 4, 0.1, (1.0, 1.0, 0.5, 0.25)),
    3: ConfigSpec("batched_decode", 2, 32, 4096, 8, 128, 32, 4, 0.05, (1.0, 1.0, 1.0, 1.0)),
    4: ConfigSpec("long_sparse", 3, 4, 32768, 8, 128, 64, 4, 0.1, (1.0, 1.0, 0.5, 0.25),
                  k_outlier_frac=0.01, k_outlier_gain=20.0),
    5: ConfigSpec("ragged_layers", 4, 64, None, 8, 128, 32, 4, 0.1, (1.0, 1.0, 0.5, 0.25),
                  ragged=(512, 16384), mixed=True, layers=24),
}


@dataclass
class Request:
    T: int
    xk: list  # per loop: BF16 [T, H, D]
    xv: list
    active: list  # per loop: int32 [n] ascending, or None (dense)


@dataclass
class Workload:
    spec: ConfigSpec
    layer: int
    H: int
    D: int
    Hq: int
    depth: int
    requests: list = field(default_factory=list)
    q: torch.Tensor | None = None  # BF16 [B, Hq, D]

    @property
    def n_requests(self) -> int:
        return len(self.requests)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed & 0x7FFFFFFFFFFFFFFF)
    return g


def request_lengths(spec: ConfigSpec) -> list:
    if spec.ragged is None:
        return [spec.T] * spec.n_requests
    g = _gen("cpu", spec.seed * 7919 + 1)
    lo, hi = spec.ragged
    out = []
    for _ in range(spec.n_requests):
        while True:
            t = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
            if t % 64 != 0:
                break
        out.append(t)
    return out


def request_is_sparse(spec: ConfigSpec) -> list:
    if not spec.mixed:
        return [any(r < 1.0 for r in spec.ratios)] * spec.n_requests
    g = _gen("cpu", spec.seed * 7919 + 2)
    return [bool(torch.randint(0, 2, (1,), generator=g).item()) for _ in range(spec.n_requests)]


def k_outlier_pairs(spec: ConfigSpec) -> list:
    """(head, channel) pairs whose base K is scaled, 1% of H*D rounded."""
    if spec.k_outlier_frac <= 0:
        return []
    n = max(1, round(spec.k_outlier_frac * spec.H * spec.D))
    g = _gen("cpu", spec.seed * 7919 + 3)
    flat = torch.randperm(spec.H * spec.D, generator=g)[:n].sort().values
    return [(int(i) // spec.D, int(i) % spec.D) for i in flat]


def _drift_chain(T, H, D, loops, sigma, g, device, gain_mask=None):
    x = torch.randn((T, H, D), generator=g, device=device, dtype=torch.float32)
    if gain_mask is not None:
        x = x * gain_mask
    out = [x.to(torch.bfloat16)]
    for _ in range(1, loops):
        x = x + sigma * torch.randn((T, H, D), generator=g, device=device, dtype=torch.float32)
        out.append(x.to(torch.bfloat16))
    return out


def _nested_sets(T, ratios, sparse, g, device):
    sets = []
    prev = None  # None = all tokens
    for r in ratios:
        if r >= 1.0 or not sparse:
            sets.append(None)
            continue
        n = min(T, math.ceil(r * T))
        pool = torch.arange(T, device=device, dtype=torch.int64) if prev is None else prev.to(torch.int64)
        pick = torch.randperm(pool.numel(), generator=g, device=device)[:n]
        cur = pool[pick].sort().values.to(torch.int32).contiguous()
        sets.append(cur)
        prev = cur
    return sets


def make_request(spec: ConfigSpec, layer: int, b: int, device="cpu", T: int | None = None,
                 sparse: bool | None = None) -> Request:
    """One request's K/V chains and active sets; reproducible per (config, layer, request)."""
    if T is None:
        T = spec.T if spec.ragged is None else request_lengths(spec)[b % spec.n_requests]
    if sparse is None:
        sparse = request_is_sparse(spec)[b % spec.n_requests]
    seed = (spec.seed + 1) * 1_000_003 + layer * 10_007 + b
    g = _gen(device, seed)
    gain = None
    pairs = k_outlier_pairs(spec)
    if pairs:
        gain = torch.ones((1, spec.H, spec.D), device=device, dtype=torch.float32)
        for h, d in pairs:
            gain[0, h, d] = spec.k_outlier_gain
    xk = _drift_chain(T, spec.H, spec.D, spec.loops, spec.sigma, g, device, gain)
    xv = _drift_chain(T, spec.H, spec.D, spec.loops, spec.sigma, g, device)
    active = _nested_sets(T, spec.ratios, sparse, g, device)
    return Request(T, xk, xv, active)


def make_queries(spec: ConfigSpec, layer: int, n_requests: int, device="cpu") -> torch.Tensor:
    g = _gen(device, (spec.seed + 1) * 1_000_003 + layer * 10_007 + 999_983)
    return torch.randn((n_requests, spec.Hq, spec.D), generator=g, device=device).to(torch.bfloat16)


def make_workload(idx: int, device="cpu", layer: int = 0, requests=None, replicate: int = 1) -> Workload:
    """Workload of configuration `idx` (1..5) for one layer.

    `requests` selects a subset of request indices (default: all). `replicate`
    > 1 builds that many independent copies of the request list, each with its
    own seed (used for the batched replicate of the single-request configs).
    """
    spec = CONFIGS[idx]
    lengths = request_lengths(spec)
    sparse = request_is_sparse(spec)
    idxs = list(range(spec.n_requests)) if requests is None else list(requests)
    reqs = []
    for rep in range(replicate):
        for b in idxs:
            rb = b + rep * spec.n_requests
            reqs.append(make_request(spec, layer, rb, device, T=lengths[b], sparse=sparse[b]))
    q = make_queries(spec, layer, len(reqs), device)
    return Workload(spec, layer, spec.H, spec.D, spec.Hq, spec.loops, reqs, q)


def bf16_bits(t: torch.Tensor):
    """BF16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")
