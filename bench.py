#!/usr/bin/env python
"""Benchmark of the packed-KV hot path on GB300.

One step = one pass of the whole path over one batch of synthetic requests:
batched encode of the loop-1 base and the loop-2..4 residuals of K and V,
batched reconstruction at depth 4 of K and V, and packed-KV GQA decode
attention at depth 4. Inputs are resident in HBM before the timed region and
larger than L2. The reported value is the metric's first quantity: the packed
decode attention's algorithmic bytes (chain payloads to the depth, q, output)
per second of its phase inside the step; encode and reconstruction GB/s and
the whole step's rate are reported beside it ("phases"). "e2e" is the same
attention through the C ABI with the packed chains and q in pinned host memory
(copied in every step) and the output read back. "configs" times the encode,
reconstruction and attention of configurations 3, 4 and 5 on their own.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the CPU oracle timed on host cores)

Multi-GPU (torchrun, one rank per GPU): every rank runs its own independent
batch (weak scaling), no data-path collective; the timed region is bracketed
by a barrier and a synchronize, and the max time over ranks is reported.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "packed-KV decode attn GB/s & % of GB300 HBM peak; encode/reconstruct GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

# name -> (configuration index, replicate count, description)
WORKLOADS = {
    "cfg2x512": (2, 512, "512 independent requests of the partial-group sparse configuration: 1000 tokens each "
                         "(tail group of 40), H=8 KV heads x D=128, Hq=32, 4 loops, loops 3/4 compact sparse over "
                         "nested random sets of 50%/25%"),
    "cfg3": (3, 1, "32 requests x 4096 tokens, H=8 x D=128, Hq=32, 4 dense loops"),
    "cfg4": (4, 1, "4 requests x 32768 tokens, H=8 x D=128, Hq=64, loops 3/4 sparse 50%/25%, 1% K outlier channels"),
    "cfg1": (1, 1, "1 request x 256 tokens, H=8 x D=128, Hq=32, 4 dense loops"),
}


CONFIG_DESCRIPTIONS = {
    "cfg3": WORKLOADS["cfg3"][2],
    "cfg4": WORKLOADS["cfg4"][2],
    "cfg5": "24 layers x 64 requests, lengths uniform 512..16384 (not multiples of 64), H=8 x D=128, Hq=32, 4 loops, "
            "per request dense or sparse 50%/25% late loops; contiguous per-request buffers and a device request table",
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="cfg2x512")
    ap.add_argument("--algo", choices=["auto", "simt", "mma", "mma_general", "tcgen05"], default="auto")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the extra timings (sparse decode, BF16 tail, tile-local K grouping)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target wall time of the CPU-oracle sample")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration timings (configs 3, 4, 5)")
    return ap.parse_args(argv)


def parse_args_list(argv):
    return parse_args(list(argv))


# ------------------------------------------------------------------ algorithmic bytes


def request_sizes(req, H):
    rows = [req.T if a is None else int(a.numel()) for a in req.active]
    sparse = [a is not None for a in req.active]
    return rows, sparse


def algorithmic_bytes(reqs, H, D, Hq, depth, payload):
    """Per-phase algorithmic bytes of one step.

    encode (loop r, K or V): read the BF16 source rows (2*n_r*H*D), read the
    predecessor chain at those rows (each earlier loop's payload scaled by
    n_r/n_j), write the loop's payload. reconstruct: read the chain payload to
    the depth, write BF16 [T, H, D]. attention: read the K and V chain payloads
    (with the shared sparse index once), q (BF16) and the FP32 output."""
    enc = rec = att = 0
    tokens = 0
    for req in reqs:
        rows, sparse = request_sizes(req, H)
        tokens += req.T
        for kind in (0, 1):
            pl = [payload(kind, rows[j], sparse[j]) for j in range(depth)]
            for r in range(depth):
                enc += 2 * rows[r] * H * D + pl[r]
                for j in range(r):
                    enc += pl[j] * (rows[r] / rows[j] if rows[j] else 0.0)
            rec += sum(pl) + 2 * req.T * H * D
        att += sum(payload(0, rows[j], sparse[j]) + payload(1, rows[j], False) for j in range(depth))
        att += 2 * Hq * D + 4 * Hq * D
    return {"encode": enc, "reconstruct": rec, "attention": att, "tokens": tokens}


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        self.gpu = ids[local_rank] if local_rank < len(ids) else str(local_rank)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_traffic(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))[kernel_key]
    except Exception:
        return None
    src = os.path.join(ROOT, d["source"])
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    if sha != d.get("source_sha"):
        return None
    return d


# ------------------------------------------------------------------ multi-rank helpers


def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank time over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, step_bytes: float, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own batch of step_bytes
    per step (weak scaling); the step time is the slowest rank's."""
    return world * step_bytes / (ms_per_step * 1e-3) / 1e9


def rank_workload(cfg_idx: int, rank: int, replicate: int, device):
    """The independent batch of one rank: same shapes on every rank, drawn from
    a rank-specific seed (the rank plays the role of the layer index)."""
    from quantized_cross_loop_gb300 import workloads as W

    return W.make_workload(cfg_idx, device=device, layer=rank, replicate=replicate)


# ------------------------------------------------------------------ CPU oracle


def oracle_attention_sample(reqs, q_rows, depth, scale, threads, outputs=None):
    """The CPU oracle's packed decode attention over `reqs` with `threads` host
    threads: the FP32 decode of the K and V chains at `depth`, then FP32
    attention. The chains are encoded first, untimed. Returns seconds; the
    outputs are appended to `outputs` when it is a list."""
    from oracle import oracle as O
    from quantized_cross_loop_gb300.workloads import bf16_bits

    import numpy as np

    def encode(i):
        req = reqs[i]
        act = [None if a is None else a.cpu().numpy().astype(np.int32) for a in req.active]
        ks = O.encode_chain(O.KIND_K, [bf16_bits(x) for x in req.xk], act)
        vs = O.encode_chain(O.KIND_V, [bf16_bits(x) for x in req.xv], act)
        return ks, vs, bf16_bits(q_rows[i])

    O.lib()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        chains = list(ex.map(encode, range(len(reqs))))
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        res = list(ex.map(lambda c: O.attention_f32(c[2], O.decode_f32(c[0], depth), O.decode_f32(c[1], depth), scale),
                          chains))
    secs = time.perf_counter() - t0
    if outputs is not None:
        outputs.extend(res)
    return secs


def attention_bytes(reqs, H, D, Hq, depth, payload):
    return algorithmic_bytes(reqs, H, D, Hq, depth, payload)["attention"]


# ------------------------------------------------------------------ main


def main():
    args = parse_args()
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg_idx, replicate, desc = WORKLOADS[args.workload]

    if args.impl == "reference":
        return run_reference(args, world, rank, cfg_idx, replicate, desc)

    from quantized_cross_loop_gb300 import build as kbuild
    from quantized_cross_loop_gb300 import kvq
    from quantized_cross_loop_gb300 import workloads as W

    if not os.path.exists(kvq.LIB_PATH):
        kbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    # ---- workload, resident in HBM (each rank its own independent batch)
    wl = rank_workload(cfg_idx, rank, replicate, dev)
    reqs = wl.requests
    src_all, src_chunks = pack_sources(reqs, torch, dev)  # one buffer in (loop, kind) chunks for the end-to-end run
    B, H, D, Hq, depth = wl.n_requests, wl.H, wl.D, wl.Hq, wl.depth
    lengths = [r.T for r in reqs]
    pool = kvq.PackedPool(lengths, [r.active for r in reqs], H, D, depth, dev)
    xk_ptrs = [kvq.pointer_array([r.xk[j] for r in reqs], dev) for j in range(depth)]
    xv_ptrs = [kvq.pointer_array([r.xv[j] for r in reqs], dev) for j in range(depth)]
    total_rows = sum(lengths)
    rk = torch.empty((total_rows, H, D), dtype=torch.bfloat16, device=dev)
    rv = torch.empty_like(rk)
    offs = [0]
    for t in lengths:
        offs.append(offs[-1] + t)
    rk_ptrs = kvq.pointer_array([rk[offs[b]:offs[b + 1]] for b in range(B)], dev)
    rv_ptrs = kvq.pointer_array([rv[offs[b]:offs[b + 1]] for b in range(B)], dev)
    q = wl.q.contiguous()
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(B, H, Hq, D), dtype=torch.uint8, device=dev)
    algo = {"auto": kvq.ATTN_AUTO, "simt": kvq.ATTN_SIMT, "mma": kvq.ATTN_MMA, "mma_general": kvq.ATTN_MMA_GENERAL,
            "tcgen05": kvq.ATTN_TCGEN05}[args.algo]
    stream = torch.cuda.current_stream()

    # K and V chains are independent: V runs on a second stream with its own
    # batch workspace, joined back at the end of each phase
    side = torch.cuda.Stream(device=dev)
    side_ws = torch.empty_like(pool.workspace)

    def fork():
        ev = torch.cuda.Event()
        ev.record(stream)
        side.wait_event(ev)

    def join():
        ev = torch.cuda.Event()
        ev.record(side)
        stream.wait_event(ev)

    def encode_all(ready=None):
        """ready[j] = (K event, V event): the sources of loop j have arrived (end-to-end run)."""
        fork()
        for j in range(depth):
            if ready is not None:
                stream.wait_event(ready[j][0])
                side.wait_event(ready[j][1])
            kvq.kvq_encode_batch(pool, kvq.KVQ_K, j, xk_ptrs[j], stream=stream)
            kvq.kvq_encode_batch(pool, kvq.KVQ_V, j, xv_ptrs[j], stream=side, workspace=side_ws)
        join()

    def reconstruct_all():
        fork()
        kvq.kvq_reconstruct_batch(pool, kvq.KVQ_K, depth, rk_ptrs, stream=stream)
        kvq.kvq_reconstruct_batch(pool, kvq.KVQ_V, depth, rv_ptrs, stream=side, workspace=side_ws)
        join()

    def attend():
        kvq.kvq_decode_attn_packed(pool.table, q, depth, H, algo=algo, out=out, workspace=ws)

    n_ev = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_ev)]

    def step(e=None, ready=None, after_encode=None):
        if e:
            e[0].record(stream)
        encode_all(ready)
        if after_encode is not None:
            after_encode.record(stream)
        if e:
            e[1].record(stream)
        reconstruct_all()
        if e:
            e[2].record(stream)
        attend()
        if e:
            e[3].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    err = kvq.attn_error_word(ws) | kvq.attn_error_word(pool.workspace) | kvq.attn_error_word(side_ws)
    if err:
        raise RuntimeError(f"error word {err}")

    clocks = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start
    launches0 = kvq.launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = kvq.launch_count() - launches0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    enc_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    rec_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    att_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps

    ab = algorithmic_bytes(reqs, H, D, Hq, depth, lambda k, n, s: kvq.payload_bytes(k, n, H, D, s))
    step_bytes = ab["encode"] + ab["reconstruct"] + ab["attention"]
    att_ms_all = max_over_ranks(att_ms, dev)
    value = whole_job_gbs(world, ab["attention"], att_ms_all)  # the metric's first quantity: packed decode attention
    peak, peak_kind = measured_peak()
    phase_ms = {"encode": enc_ms, "reconstruct": rec_ms, "attention": att_ms}
    phase_gbs = {k: ab[k] / (phase_ms[k] * 1e-3) / 1e9 for k in phase_ms}

    # ---- end to end through the public API with host buffers: the attention
    # with the packed chains and q copied from host memory every step; beside
    # it, the whole path with the BF16 sources copied in
    e2e = e2e_whole = None
    if not args.no_e2e:
        e2e = run_e2e_attention(args, torch, kvq, pool, q, out, attend, stream, world, dev, ab["attention"], dist)
        e2e_whole = run_e2e(args, torch, kvq, src_all, src_chunks, q, out, step, stream, world, dev, step_bytes, dist)

    # ---- roofline of the attention kernel call (plan + attention + combine)
    dominant = max(phase_ms, key=phase_ms.get)
    att_key = {kvq.ATTN_AUTO: "attn_auto", kvq.ATTN_SIMT: "attn_simt", kvq.ATTN_MMA: "attn_mma",
               kvq.ATTN_MMA_GENERAL: "attn_mma_general", kvq.ATTN_TCGEN05: "attn_tcgen05"}[algo]
    tr = kernel_traffic(att_key)
    traffic = None
    if tr is not None and tr.get("workload") == args.workload:
        traffic = tr["dram_bytes_per_launch"]
    roof = {"bound": "hbm", "kernel": "kvq_decode_attn_packed (" + args.algo + ")", "achieved": phase_gbs["attention"],
            "peak": peak, "unit": "GB/s", "frac": phase_gbs["attention"] / peak, "peak_source": peak_kind,
            "frac_of_nominal_8tbs": phase_gbs["attention"] / NOMINAL_HBM_GBS, "traffic": traffic,
            "algorithmic_bytes_per_launch": ab["attention"], "avg_launch_ms": att_ms,
            "dominant_phase_of_step": dominant}

    extras = None
    if not args.no_extras:
        extras = run_extras(torch, kvq, pool, reqs, q, H, Hq, D, depth, dev, stream,
                            (xk_ptrs, xv_ptrs, rk_ptrs, rv_ptrs, rk, rv, offs))

    configs = None
    if world == 1 and not args.no_configs:
        configs = run_configs(torch, kvq, dev, stream, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gpu_out = kvq.kvq_decode_attn_packed(pool.table, q, depth, H, algo=algo, workspace=ws).cpu().numpy()
        cpu = run_cpu_baseline(args, reqs, q, depth, D, H, Hq, kvq, gpu_out)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded, generated on the device)",
            "config": {"workload": args.workload, "description": desc, "requests_per_gpu": B,
                       "tokens_per_request": "ragged" if len(set(lengths)) > 1 else lengths[0], "kv_heads": H,
                       "head_dim": D, "q_heads": Hq, "loops": depth, "attn_kernel": args.algo,
                       "l2": "inputs larger than L2 (BF16 sources %.1f GB, packed %.2f GB per GPU), no flush"
                             % (sum(2 * r.T * H * D * 2 * depth for r in reqs) / 1e9, pool.payload_bytes / 1e9),
                       "arithmetic": "codec FP32 with BF16/FP16 rounding (bit-exact), attention FP32 accumulate",
                       "parallelism": f"replicas x{world} (independent batches, no collective)",
                       "streams": "K chain on the launching stream, V chain on a second stream, joined per phase"},
            "phases": {"whole_step_gbs": whole_job_gbs(world, step_bytes, ms_per_step),
                       "encode_gbs": phase_gbs["encode"], "reconstruct_gbs": phase_gbs["reconstruct"],
                       "attention_gbs": phase_gbs["attention"], "encode_ms": enc_ms, "reconstruct_ms": rec_ms,
                       "attention_ms": att_ms, "attention_pct_of_measured_hbm": 100 * phase_gbs["attention"] / peak,
                       "attention_pct_of_8tbs": 100 * phase_gbs["attention"] / NOMINAL_HBM_GBS,
                       "attended_tokens_per_s": ab["tokens"] / (att_ms * 1e-3),
                       "encoded_tokens_per_s": ab["tokens"] / (enc_ms * 1e-3)},
            "roofline": roof,
            "configs": configs,
            "extras": extras,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "e2e_whole_path": e2e_whole,
            "clocks": clk,
            "gpu_launches": launches,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def pack_sources(reqs, torch, dev):
    """Moves every request's BF16 sources into one device buffer (the
    requests' tensors become views of it), ordered by loop, then K before V,
    then request, so that the sources of one (loop, kind) are one contiguous
    chunk. Returns the buffer and the chunks' element ranges [loop][kind]."""
    total = sum(x.numel() for r in reqs for xs in (r.xk, r.xv) for x in xs)
    flat = torch.empty(total, dtype=torch.bfloat16, device=dev)
    depth = len(reqs[0].xk) if reqs else 0
    off = 0
    chunks = []
    for j in range(depth):
        per_kind = []
        for kind in (0, 1):
            start = off
            for r in reqs:
                xs = r.xk if kind == 0 else r.xv
                v = flat[off:off + xs[j].numel()].view(xs[j].shape)
                v.copy_(xs[j])
                xs[j] = v
                off += v.numel()
            per_kind.append((start, off))
        chunks.append(per_kind)
    torch.cuda.synchronize()
    return flat, chunks


def run_extras(torch, kvq, pool, reqs, q, H, Hq, D, depth, dev, stream, ptrs, reps=10):
    """Timings of the variants next to the step, on the same workload (CUDA
    events, after one warm-up call each):
      sparse decode attention (RFC §3.2): reference state at loop 2 keeping a
      quarter of each request's keys per query head, then one later loop at
      the full depth reading only those keys;
      dense attention with a 100-token BF16 tail per request (RFC §3.3);
      tile-local K grouping (codec PR review, group ownership vs pages): the
      K encode, K reconstruction and attention of a second pool whose sparse
      K groups stay inside one 64-token tile, beside the K phases of the
      compact-grouped pool;
      NVFP4 residual loops (codec PR review: INT4 base + NVFP4 residuals,
      compared on fused-attention speed and accuracy): encode, reconstruction
      and attention of a pool whose loops 2.. are NVFP4, beside the INT4 pool
      on one stream, and the accuracy of both on a sample of requests against
      the unquantised chain (each token's BF16 source from the deepest loop
      that stores it, which is what the chain reconstructs): reconstruction
      RMS error, and the attention error against FP32 attention over it."""
    B = len(reqs)
    max_t = max(r.T for r in reqs)
    n_select = max(1, max_t // 4)
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    q2 = torch.randn(q.shape, generator=g, device=dev).to(torch.bfloat16)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            r = fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps, r

    ref_ms, st = timed(lambda: kvq.kvq_sparse_ref_state(pool.table, q2, 2, H, n_select, max_t))
    dec_ws = torch.zeros(kvq.kvq_sparse_decode_workspace_bytes(B, H, Hq, D, max_t), dtype=torch.uint8, device=dev)
    dec_ms, _ = timed(lambda: kvq.kvq_sparse_decode_attn(pool.table, q, depth, H, st, workspace=dec_ws,
                                                         algo=kvq.ATTN_MMA))
    pk_ws = torch.zeros(16, dtype=torch.uint8, device=dev)  # the per-key gather kernel
    pk_ms, _ = timed(lambda: kvq.kvq_sparse_decode_attn(pool.table, q, depth, H, st, workspace=pk_ws,
                                                        algo=kvq.ATTN_SIMT))
    err = kvq.attn_error_word(st.workspace) | kvq.attn_error_word(dec_ws) | kvq.attn_error_word(pk_ws)
    selected = sum(min(n_select, r.T) for r in reqs) * Hq
    # budget sweep: the later loop by both kernels against the dense attention at the same depth
    dws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(B, H, Hq, D), dtype=torch.uint8, device=dev)
    dense_ms, _ = timed(lambda: kvq.kvq_decode_attn_packed(pool.table, q, depth, H, workspace=dws))
    err |= kvq.attn_error_word(dws)
    sweep = []
    for frac in (0.01, 0.025, 0.05, 0.1, 0.25):
        ns = max(1, int(round(frac * max_t)))
        rs_ms, sst = timed(lambda: kvq.kvq_sparse_ref_state(pool.table, q2, 2, H, ns, max_t))
        m_ms, _ = timed(lambda: kvq.kvq_sparse_decode_attn(pool.table, q, depth, H, sst, workspace=dec_ws,
                                                           algo=kvq.ATTN_MMA))
        g_ms, _ = timed(lambda: kvq.kvq_sparse_decode_attn(pool.table, q, depth, H, sst, workspace=pk_ws,
                                                           algo=kvq.ATTN_SIMT))
        a_ms, _ = timed(lambda: kvq.kvq_sparse_decode_attn(pool.table, q, depth, H, sst, workspace=dec_ws))
        err |= kvq.attn_error_word(sst.workspace) | kvq.attn_error_word(dec_ws) | kvq.attn_error_word(pk_ws)
        sweep.append({"keys_per_query_head": ns, "fraction": frac, "ref_state_ms": rs_ms,
                      "later_loop_masked_ms": m_ms, "later_loop_gather_ms": g_ms, "later_loop_auto_ms": a_ms,
                      "later_loop_vs_dense": min(m_ms, g_ms) / dense_ms})
        del sst
    empty = torch.zeros((0, H, D), dtype=torch.bfloat16, device=dev)
    tail = [(empty, empty, torch.randn((100, H, D), generator=g, device=dev).to(torch.bfloat16),
             torch.randn((100, H, D), generator=g, device=dev).to(torch.bfloat16)) for _ in reqs]
    ks = [pool.k_streams[b] for b in range(B)]
    vs = [pool.v_streams[b] for b in range(B)]
    ttable = kvq.RequestTable(ks, vs, dev, segments=tail)
    tws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(B, H, Hq, D), dtype=torch.uint8, device=dev)
    tail_ms, _ = timed(lambda: kvq.kvq_decode_attn_packed(ttable, q, depth, H, workspace=tws))
    err |= kvq.attn_error_word(tws)

    xk_ptrs, xv_ptrs, rk_ptrs, rv_ptrs, rk, rv, offs = ptrs
    tpool = kvq.PackedPool([r.T for r in reqs], [r.active for r in reqs], H, D, depth, dev, kgroup=kvq.KVQ_KGROUP_TILE)

    def enc_k(pl):
        for j in range(depth):
            kvq.kvq_encode_batch(pl, kvq.KVQ_K, j, xk_ptrs[j], stream=stream)

    for j in range(depth):
        kvq.kvq_encode_batch(tpool, kvq.KVQ_V, j, xv_ptrs[j], stream=stream)
    ek_t, _ = timed(lambda: enc_k(tpool))
    ek_c, _ = timed(lambda: enc_k(pool))
    rk_t, _ = timed(lambda: kvq.kvq_reconstruct_batch(tpool, kvq.KVQ_K, depth, rk_ptrs, stream=stream))
    rk_c, _ = timed(lambda: kvq.kvq_reconstruct_batch(pool, kvq.KVQ_K, depth, rk_ptrs, stream=stream))
    kws = torch.empty_like(tws)
    at_t, _ = timed(lambda: kvq.kvq_decode_attn_packed(tpool.table, q, depth, H, workspace=kws))
    err |= kvq.attn_error_word(kws) | kvq.attn_error_word(tpool.workspace)
    kgroup_tile = {"payload_bytes": tpool.payload_bytes, "payload_bytes_compact": pool.payload_bytes,
                   "encode_k_ms": ek_t, "encode_k_ms_compact": ek_c,
                   "reconstruct_k_ms": rk_t, "reconstruct_k_ms_compact": rk_c, "attention_ms": at_t}
    del tpool
    nvfp4 = run_nvfp4_extra(torch, kvq, pool, reqs, q, H, Hq, D, depth, dev, stream, timed, ptrs)
    err |= nvfp4.pop("error_word")
    append = run_append_extra(torch, kvq, reqs, H, D, depth, dev, stream)
    return {"kgroup_tile": kgroup_tile, "nvfp4_residuals": nvfp4, "append_tile": append,
            "sparse_decode": {"budget_keys_per_query_head": n_select, "ref_depth": 2, "depth": depth,
                              "ref_state_ms": ref_ms, "later_loop_ms": dec_ms,
                              "later_loop_kernel": "key-masked tensor-core attention",
                              "later_loop_ms_per_key_kernel": pk_ms,
                              "selected_keys_per_s": selected / (dec_ms * 1e-3),
                              "dense_attention_ms": dense_ms, "budget_sweep": sweep},
            "bf16_tail": {"tail_tokens_per_request": 100, "attention_ms": tail_ms},
            "error_word": err}


def run_append_extra(torch, kvq, reqs, H, D, depth, dev, stream, reps=5):
    """Cost of the tail flush (RFC §3.3): one 64-token tile appended to the K and V
    chains of every request in one batched call (kvq_append_tile_batch), on a pool
    of growable chains (tile-local K grouping) holding each request's tokens up to
    its last whole tile but one; `reps` fresh pools are timed and averaged."""
    from quantized_cross_loop_gb300.kvq import KVQ_KGROUP_TILE
    B = len(reqs)
    T0 = [(r.T // 64 - 1) * 64 for r in reqs]
    act0 = [[None if a is None else a[a < T0[b]].contiguous() for a in reqs[b].active] for b in range(B)]
    xk = [[reqs[b].xk[j][T0[b]:T0[b] + 64].contiguous() for b in range(B)] for j in range(depth)]
    xv = [[reqs[b].xv[j][T0[b]:T0[b] + 64].contiguous() for b in range(B)] for j in range(depth)]
    rel = [[None if reqs[b].active[j] is None else
            (reqs[b].active[j][(reqs[b].active[j] >= T0[b]) & (reqs[b].active[j] < T0[b] + 64)] - T0[b]).to(torch.int32)
            for b in range(B)] for j in range(depth)]
    src = [[kvq.pointer_array([reqs[b].xk[j] for b in range(B)], dev) for j in range(depth)],
           [kvq.pointer_array([reqs[b].xv[j] for b in range(B)], dev) for j in range(depth)]]
    total, err = 0.0, 0
    for _ in range(reps):
        pool = kvq.PackedPool(T0, act0, H, D, depth, dev, kgroup=KVQ_KGROUP_TILE, token_caps=[t + 64 for t in T0])
        for j in range(depth):
            kvq.kvq_encode_batch(pool, kvq.KVQ_K, j, src[0][j], stream=stream)
            kvq.kvq_encode_batch(pool, kvq.KVQ_V, j, src[1][j], stream=stream)
        ws = torch.empty(int(kvq.lib().kvq_append_batch_workspace_bytes(B)), dtype=torch.uint8, device=dev)
        pool.append_tile(xk, xv, rel, workspace=ws, stream=stream)  # warm-up call
        torch.cuda.synchronize()
        err |= kvq.attn_error_word(ws)
        pool2 = kvq.PackedPool(T0, act0, H, D, depth, dev, kgroup=KVQ_KGROUP_TILE, token_caps=[t + 64 for t in T0])
        for j in range(depth):
            kvq.kvq_encode_batch(pool2, kvq.KVQ_K, j, src[0][j], stream=stream)
            kvq.kvq_encode_batch(pool2, kvq.KVQ_V, j, src[1][j], stream=stream)
        prep = pool2.prepare_append(xk, xv, rel)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pool2.append_tile(workspace=ws, stream=stream, prepared=prep)
        b.record(stream)
        torch.cuda.synchronize()
        total += a.elapsed_time(b)
        err |= kvq.attn_error_word(ws)
        del pool, pool2
    ms = total / reps
    return {"requests": B, "tokens_per_request": 64, "ms_per_call": ms, "us_per_request_k_and_v": ms * 1e3 / B,
            "launches": 3 + 4 * depth, "error_word": err}


def run_nvfp4_extra(torch, kvq, pool, reqs, q, H, Hq, D, depth, dev, stream, timed, ptrs, n_sample=16):
    """INT4-base + NVFP4-residual chains against the INT4 chains of `pool` (see run_extras)."""
    xk_ptrs, xv_ptrs, rk_ptrs, rv_ptrs, rk, rv, offs = ptrs
    formats = [kvq.KVQ_FMT_INT4] + [kvq.KVQ_FMT_NVFP4] * (depth - 1)
    npool = kvq.PackedPool([r.T for r in reqs], [r.active for r in reqs], H, D, depth, dev, formats=formats)

    def enc(pl):
        for j in range(depth):
            kvq.kvq_encode_batch(pl, kvq.KVQ_K, j, xk_ptrs[j], stream=stream)
            kvq.kvq_encode_batch(pl, kvq.KVQ_V, j, xv_ptrs[j], stream=stream)

    def rec(pl):
        kvq.kvq_reconstruct_batch(pl, kvq.KVQ_K, depth, rk_ptrs, stream=stream)
        kvq.kvq_reconstruct_batch(pl, kvq.KVQ_V, depth, rv_ptrs, stream=stream)

    B = len(reqs)
    ws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(B, H, Hq, D), dtype=torch.uint8, device=dev)
    out_n = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    out_i = torch.empty_like(out_n)
    enc_n, _ = timed(lambda: enc(npool))
    enc_i, _ = timed(lambda: enc(pool))
    rec_i, _ = timed(lambda: rec(pool))
    sample = list(range(min(n_sample, B)))
    rmse = {}

    def target(xs, act):  # the unquantised chain: a token keeps the source of the deepest loop storing it
        t = xs[0].clone()
        for j in range(1, depth):
            if act[j] is None:
                t = xs[j].clone()
            else:
                t[act[j].long()] = xs[j][act[j].long()]
        return t

    tk = {b: target(reqs[b].xk, reqs[b].active) for b in sample}
    tv = {b: target(reqs[b].xv, reqs[b].active) for b in sample}

    def recon_rmse(tag):
        for kind, buf, src in (("k", rk, tk), ("v", rv, tv)):
            num = den = 0.0
            for b in sample:
                d = buf[offs[b]:offs[b + 1]].float() - src[b].float()
                num += float((d * d).sum())
                den += d.numel()
            rmse[f"{kind}_{tag}"] = (num / max(den, 1)) ** 0.5

    recon_rmse("int4")
    rec_n, _ = timed(lambda: rec(npool))
    recon_rmse("nvfp4")
    att_n, _ = timed(lambda: kvq.kvq_decode_attn_packed(npool.table, q, depth, H, out=out_n, workspace=ws))
    att_i, _ = timed(lambda: kvq.kvq_decode_attn_packed(pool.table, q, depth, H, out=out_i, workspace=ws))
    # the NVFP4-reading form of the tensor-core kernel on the INT4 pool: the cost of carrying both formats
    att_in, _ = timed(lambda: kvq.kvq_decode_attn_packed(pool.table, q, depth, H,
                                                         algo=kvq.ATTN_MMA_GENERAL | kvq.ATTN_NVFP4,
                                                         out=out_i, workspace=ws))
    # the INT4 pool called with the NVFP4 flag: the plan finds no NVFP4 loop and the INT4 kernel runs
    att_if, _ = timed(lambda: kvq.kvq_decode_attn_packed(pool.table, q, depth, H, algo=kvq.ATTN_AUTO | kvq.ATTN_NVFP4,
                                                         out=out_i, workspace=ws))
    err = kvq.attn_error_word(ws) | kvq.attn_error_word(npool.workspace)
    # attention error against FP32 attention over the unquantised chain
    g = Hq // H
    scale = 1.0 / math.sqrt(D)
    worst = {"int4": 0.0, "nvfp4": 0.0}
    for b in sample:
        kx, vx = tk[b].float(), tv[b].float()  # [T, H, D]
        qb = q[b].float().view(H, g, D)
        s_ = torch.einsum("hgd,thd->hgt", qb, kx) * scale
        ref = torch.einsum("hgt,thd->hgd", torch.softmax(s_, dim=-1), vx).reshape(Hq, D)
        worst["int4"] = max(worst["int4"], float((out_i[b] - ref).abs().max()))
        worst["nvfp4"] = max(worst["nvfp4"], float((out_n[b] - ref).abs().max()))
    res = {"formats": "INT4 base, NVFP4 loops 2..%d" % depth, "payload_bytes": npool.payload_bytes,
           "payload_bytes_int4": pool.payload_bytes, "encode_ms": enc_n, "encode_ms_int4": enc_i,
           "reconstruct_ms": rec_n, "reconstruct_ms_int4": rec_i, "attention_ms": att_n, "attention_ms_int4": att_i,
           "attention_ms_int4_in_nvfp4_form": att_in, "attention_ms_int4_with_nvfp4_flag": att_if,
           "sample_requests": len(sample),
           "recon_rmse_vs_unquantised_chain": rmse, "attn_max_abs_err_vs_unquantised_chain": worst,
           "error_word": err}
    del npool
    return res


def run_e2e(args, torch, kvq, src_all, src_chunks, q, out, step, stream, world, dev, step_bytes, dist):
    """Same step through the public API with host inputs: H2D of every BF16
    source (one pinned buffer) and of q, the step, D2H of the attention output.
    The sources move in (loop, kind) chunks on a copy stream, and each loop's
    encode waits only for its own chunk, so the copies of later loops overlap
    the encode of earlier ones (and the next step's copies the reconstruction
    and attention of this one, once this step's encode has read its sources)."""
    host_src = torch.empty(src_all.shape, dtype=src_all.dtype, pin_memory=True).copy_(src_all)
    host_q = torch.empty(q.shape, dtype=q.dtype, pin_memory=True).copy_(q)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = host_src.numel() * host_src.element_size() + host_q.numel() * host_q.element_size()
    d2h = host_out.numel() * host_out.element_size()
    copy_s = torch.cuda.Stream(device=dev)
    sources_free = torch.cuda.Event()  # the previous step's encode has read the sources
    sources_free.record(stream)

    def e2e_step():
        copy_s.wait_event(sources_free)
        ready = []
        for per_kind in src_chunks:
            evs = []
            for (lo, hi) in per_kind:
                with torch.cuda.stream(copy_s):
                    src_all[lo:hi].copy_(host_src[lo:hi], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_s)
                evs.append(ev)
            ready.append(tuple(evs))
        q.copy_(host_q, non_blocking=True)
        step(ready=ready, after_encode=sources_free)
        host_out.copy_(out, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    n = max(3, args.steps // 10)
    if world > 1:
        dist.barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    sources_free.record(stream)  # the copies start inside the timed region
    for _ in range(n):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / n, dev)
    return {"value": whole_job_gbs(world, step_bytes, ms), "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n}


def run_e2e_attention(args, torch, kvq, pool, q, out, attend, stream, world, dev, att_bytes, dist):
    """The headline metric end to end through the public API with host buffers:
    every step copies the packed K/V chains (the pool's storage, one pinned
    host buffer) and q from host memory, runs the packed decode attention and
    reads the output back."""
    host_pool = torch.empty(pool.storage.shape, dtype=torch.uint8, pin_memory=True).copy_(pool.storage)
    host_q = torch.empty(q.shape, dtype=q.dtype, pin_memory=True).copy_(q)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = host_pool.numel() + host_q.numel() * host_q.element_size()
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        pool.storage.copy_(host_pool, non_blocking=True)
        q.copy_(host_q, non_blocking=True)
        attend()
        host_out.copy_(out, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    n = max(3, args.steps // 10)
    if world > 1:
        dist.barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / n, dev)
    return {"value": whole_job_gbs(world, att_bytes, ms), "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "path": "pinned host packed chains + q -> kvq_decode_attn_packed -> pinned host output"}


def phase_times(torch, kvq, wl, dev, stream, reps):
    """Encode (every loop of K and V), reconstruction (K and V at full depth)
    and packed decode attention of one workload resident on the device, on one
    stream: mean ms per call of each phase over `reps` calls after one warm-up
    call (the workload's data exceed L2). Returns (ms per phase, algorithmic
    bytes, error word)."""
    reqs = wl.requests
    B, H, D, Hq, depth = wl.n_requests, wl.H, wl.D, wl.Hq, wl.depth
    lengths = [r.T for r in reqs]
    pool = kvq.PackedPool(lengths, [r.active for r in reqs], H, D, depth, dev)
    xk_ptrs = [kvq.pointer_array([r.xk[j] for r in reqs], dev) for j in range(depth)]
    xv_ptrs = [kvq.pointer_array([r.xv[j] for r in reqs], dev) for j in range(depth)]
    offs = [0]
    for t in lengths:
        offs.append(offs[-1] + t)
    rk = torch.empty((offs[-1], H, D), dtype=torch.bfloat16, device=dev)
    rv = torch.empty_like(rk)
    rk_ptrs = kvq.pointer_array([rk[offs[b]:offs[b + 1]] for b in range(B)], dev)
    rv_ptrs = kvq.pointer_array([rv[offs[b]:offs[b + 1]] for b in range(B)], dev)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(B, H, Hq, D), dtype=torch.uint8, device=dev)

    def enc():
        for j in range(depth):
            kvq.kvq_encode_batch(pool, kvq.KVQ_K, j, xk_ptrs[j], stream=stream)
            kvq.kvq_encode_batch(pool, kvq.KVQ_V, j, xv_ptrs[j], stream=stream)

    def rec():
        kvq.kvq_reconstruct_batch(pool, kvq.KVQ_K, depth, rk_ptrs, stream=stream)
        kvq.kvq_reconstruct_batch(pool, kvq.KVQ_V, depth, rv_ptrs, stream=stream)

    def att():
        kvq.kvq_decode_attn_packed(pool.table, wl.q, depth, H, out=out, workspace=ws)

    ms = {}
    for name, fn in (("encode", enc), ("reconstruct", rec), ("attention", att)):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms[name] = e0.elapsed_time(e1) / reps
    err = kvq.attn_error_word(ws) | kvq.attn_error_word(pool.workspace)
    ab = algorithmic_bytes(reqs, H, D, Hq, depth, lambda k, n, sp: kvq.payload_bytes(k, n, H, D, sp))
    return ms, ab, err


def run_configs(torch, kvq, dev, stream, peak):
    """Encode, reconstruction and attention throughput of the other synthetic
    configurations, each on its own (timed in this run): 32 x 4096
    dense, 4 x 32768 sparse GQA 8, and the 24-layer ragged sweep (64 requests
    per layer, generated, encoded, timed and freed layer by layer; bytes and
    times summed over the layers)."""
    from quantized_cross_loop_gb300 import workloads as W

    res = {}
    for name, idx, layers, reps in (("cfg3", 3, 1, 10), ("cfg4", 4, 1, 10), ("cfg5", 5, 24, 3)):
        tot_ms = {"encode": 0.0, "reconstruct": 0.0, "attention": 0.0}
        tot_b = {"encode": 0.0, "reconstruct": 0.0, "attention": 0.0, "tokens": 0}
        err = 0
        for layer in range(layers):
            wl = W.make_workload(idx, device=dev, layer=layer)
            ms, ab, e = phase_times(torch, kvq, wl, dev, stream, reps)
            err |= e
            for k in tot_ms:
                tot_ms[k] += ms[k]
            for k in tot_b:
                tot_b[k] += ab[k]
            spec = wl.spec
            del wl
            torch.cuda.empty_cache()
        gbs = {k: tot_b[k] / (tot_ms[k] * 1e-3) / 1e9 for k in tot_ms}
        res[name] = {
            "description": CONFIG_DESCRIPTIONS[name], "layers": layers,
            "requests_per_layer": spec.n_requests,
            "attention_gbs": gbs["attention"], "attention_frac": gbs["attention"] / peak,
            "attention_frac_of_8tbs": gbs["attention"] / NOMINAL_HBM_GBS, "attention_ms": tot_ms["attention"],
            "attended_tokens_per_s": tot_b["tokens"] / (tot_ms["attention"] * 1e-3),
            "encode_gbs": gbs["encode"], "encode_frac": gbs["encode"] / peak, "encode_ms": tot_ms["encode"],
            "encoded_tokens_per_s": tot_b["tokens"] / (tot_ms["encode"] * 1e-3),
            "reconstruct_gbs": gbs["reconstruct"], "reconstruct_frac": gbs["reconstruct"] / peak,
            "reconstruct_ms": tot_ms["reconstruct"],
            "reconstructed_tokens_per_s": tot_b["tokens"] / (tot_ms["reconstruct"] * 1e-3),
            "algorithmic_bytes": {k: tot_b[k] for k in ("encode", "reconstruct", "attention")},
            "timing": f"mean of {reps} calls per phase after one warm-up, one stream, data larger than L2",
            "error_word": err}
    return res


def run_cpu_baseline(args, reqs, q, depth, D, H, Hq, kvq, gpu_out=None):
    """The CPU oracle's packed decode attention as it stands, on the host cores,
    over a bounded sample of the same requests; same metric and unit. With the
    GPU attention output of those requests (gpu_out), the largest absolute and
    relative differences to the oracle's output on the sample as well."""
    import numpy as np

    cores = os.cpu_count() or 1
    scale = 1.0 / math.sqrt(D)
    t1 = oracle_attention_sample(reqs[:1], q[:1], depth, scale, 1)
    n = max(1, min(len(reqs), int(args.cpu_seconds * cores / max(t1, 1e-3))))
    sample = reqs[:n]
    ref = []
    secs = oracle_attention_sample(sample, q[:n], depth, scale, cores, ref)
    accuracy = None
    if gpu_out is not None:
        r = np.stack([np.asarray(x, dtype=np.float64) for x in ref])
        g = np.asarray(gpu_out[:n], dtype=np.float64).reshape(r.shape)
        err = np.abs(g - r)
        big = np.abs(r) >= 0.05  # relative error where it means something
        accuracy = {"requests": n, "max_abs": float(err.max()),
                    "max_rel_where_abs_ref_ge_0.05": float((err[big] / np.abs(r[big])).max()) if big.any() else None,
                    "max_share_of_tolerance": float((err / (2e-3 + 1e-2 * np.abs(r))).max()),
                    "tolerance": "|gpu - oracle| <= 2e-3 + 1e-2 |oracle| per element"}

    def bytes_of(rs):
        return attention_bytes(rs, H, D, Hq, depth, lambda k, nn, s: kvq.payload_bytes(k, nn, H, D, s))

    return {"value": bytes_of(sample) / secs / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "value_1_thread": bytes_of(reqs[:1]) / t1 / 1e9, "cpu_model": cpu_model(),
            "sample": f"{n} of {len(reqs)} requests of the same workload: packed decode attention at depth {depth} "
                      f"(FP32 decode of the K/V chains, FP32 attention; chains encoded beforehand, untimed), "
                      f"{secs:.2f} s on {cores} threads; value_1_thread: one request on one thread, {t1:.3f} s",
            "gpu_vs_oracle": accuracy}


def cpu_model():
    """The host CPU as lscpu names it, else as /proc/cpuinfo does (model name, or
    implementer and part on Arm)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return platform.machine()
    fields = {}
    for line in info:
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return platform.machine()


def run_reference(args, world, rank, cfg_idx, replicate, desc):
    """--impl reference: the CPU oracle's packed decode attention timed on the
    host cores, each step a bounded sample of the same workload (rank 0 only
    under torchrun)."""
    if world > 1 and rank != 0:
        return
    from quantized_cross_loop_gb300 import workloads as W

    cores = os.cpu_count() or 1
    spec = W.CONFIGS[cfg_idx]
    n = min(4 * cores, spec.n_requests * replicate)
    if replicate > 1:
        wl = W.make_workload(cfg_idx, device="cpu", replicate=math.ceil(n / spec.n_requests))
    else:
        wl = W.make_workload(cfg_idx, device="cpu", requests=list(range(n)))
    reqs = wl.requests[:n]
    q = wl.q[:n]
    H, D, Hq, depth = wl.H, wl.D, wl.Hq, wl.depth
    scale = 1.0 / math.sqrt(D)

    def payload(kind, nn, sparse):
        from oracle import oracle as O

        return O.stream_bytes(kind, nn, H, D, sparse=sparse)

    for _ in range(args.warmup):
        oracle_attention_sample(reqs[:1], q[:1], depth, scale, 1)
    times = [oracle_attention_sample(reqs, q, depth, scale, cores) for _ in range(args.steps)]
    tot = attention_bytes(reqs, H, D, Hq, depth, payload)
    ms = 1e3 * sum(times) / len(times)
    value = tot / (ms * 1e-3) / 1e9
    sample = (f"{n} requests of {args.workload} per step: packed decode attention at depth {depth} (FP32 decode "
              f"of the chains, FP32 attention; chains encoded beforehand, untimed) on {cores} threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "description": desc, "oracle_requests_per_step": n},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


if __name__ == "__main__":
    main()
