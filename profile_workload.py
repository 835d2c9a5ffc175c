"""Runs one stage of the packed-KV path on a seeded synthetic workload, for
profilers (ncu captures of a single kernel). It reports no timing.

  python profile_workload.py --workload cfg3 --stage attention --reps 2
  python profile_workload.py --workload cfg2x128 --stage encode

Workloads: cfg1..cfg4 (the synthetic configurations), cfg2xN (N independent
requests of configuration 2). Stages:
  encode       batched encode of every loop of K and V (the sources are freed
               before the other stages run);
  reconstruct  batched reconstruction of K and V at full depth, `reps` times;
  attention    packed decode attention at full depth, `reps` times, with a
               256 MiB buffer written between calls so that every call starts
               with a cold L2;
  sparse       sparse decode attention: the reference state at loop 2 keeping a
               quarter of the keys per query head, then the full-depth loop,
               `reps` times each;
  tail         packed decode attention with a 100-token BF16 tail per request,
               `reps` times.
--kgroup tile builds the K chains with tile-local K groups (the stored rows of
one 64-token logical tile per group) instead of 64 consecutive stored rows;
--residual nvfp4 encodes loops 2.. of K and V as NVFP4 (INT4 base).
Every stage first encodes the workload (the launches a capture should skip:
2 + 4 (loops - 1) per kind, plus one per reconstruct or attention call before
the one captured).
"""

from __future__ import annotations

import argparse

import torch

from quantized_cross_loop_gb300 import kvq
from quantized_cross_loop_gb300 import workloads as W


def parse_workload(name: str):
    if name.startswith("cfg2x"):
        return 2, int(name[5:])
    return int(name[3:]), 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="cfg3")
    ap.add_argument("--stage", choices=["encode", "reconstruct", "attention", "sparse", "tail"], default="attention")
    ap.add_argument("--algo", choices=["auto", "simt", "mma", "mma_general", "tcgen05"], default="auto")
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--kgroup", choices=["compact", "tile"], default="compact")
    ap.add_argument("--residual", choices=["int4", "nvfp4"], default="int4")
    args = ap.parse_args()
    cfg, rep = parse_workload(args.workload)
    dev = torch.device("cuda")
    wl = W.make_workload(cfg, device=dev, replicate=rep)
    reqs = wl.requests
    kgroup = kvq.KVQ_KGROUP_TILE if args.kgroup == "tile" else kvq.KVQ_KGROUP_COMPACT
    formats = None
    if args.residual == "nvfp4":
        formats = [kvq.KVQ_FMT_INT4] + [kvq.KVQ_FMT_NVFP4] * (wl.depth - 1)
    pool = kvq.PackedPool([r.T for r in reqs], [r.active for r in reqs], wl.H, wl.D, wl.depth, dev, kgroup=kgroup,
                          formats=formats)
    for j in range(wl.depth):
        kvq.kvq_encode_batch(pool, kvq.KVQ_K, j, kvq.pointer_array([r.xk[j] for r in reqs], dev))
        kvq.kvq_encode_batch(pool, kvq.KVQ_V, j, kvq.pointer_array([r.xv[j] for r in reqs], dev))
    lengths = [r.T for r in reqs]
    del reqs, wl.requests[:]
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if args.stage == "reconstruct":
        outs = [[torch.empty((t, wl.H, wl.D), dtype=torch.bfloat16, device=dev) for t in lengths] for _ in range(2)]
        ptrs = [kvq.pointer_array(o, dev) for o in outs]
        for _ in range(args.reps):
            for kind in (kvq.KVQ_K, kvq.KVQ_V):
                kvq.kvq_reconstruct_batch(pool, kind, wl.depth, ptrs[kind])
    elif args.stage == "attention":
        algo = {"auto": kvq.ATTN_AUTO, "simt": kvq.ATTN_SIMT, "mma": kvq.ATTN_MMA,
                "mma_general": kvq.ATTN_MMA_GENERAL, "tcgen05": kvq.ATTN_TCGEN05}[args.algo]
        q = wl.q
        out = torch.empty(q.shape, dtype=torch.float32, device=dev)
        ws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(q.shape[0], wl.H, wl.Hq, wl.D), dtype=torch.uint8,
                         device=dev)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        for _ in range(args.reps):
            flush.zero_()
            kvq.kvq_decode_attn_packed(pool.table, q, wl.depth, wl.H, algo=algo, out=out, workspace=ws)
    elif args.stage == "sparse":
        max_t = max(lengths)
        n_select = max(1, max_t // 4)
        for _ in range(args.reps):
            st = kvq.kvq_sparse_ref_state(pool.table, wl.q, 2, wl.H, n_select, max_t)
        ws = torch.zeros(16, dtype=torch.uint8, device=dev)  # the per-key kernel, then the tensor-core path
        for _ in range(args.reps):
            kvq.kvq_sparse_decode_attn(pool.table, wl.q, wl.depth, wl.H, st, workspace=ws)
        for _ in range(args.reps):
            kvq.kvq_sparse_decode_attn(pool.table, wl.q, wl.depth, wl.H, st)
    elif args.stage == "tail":
        empty = torch.zeros((0, wl.H, wl.D), dtype=torch.bfloat16, device=dev)
        g = torch.Generator(device=dev)
        g.manual_seed(7)
        tail = [(empty, empty, torch.randn((100, wl.H, wl.D), generator=g, device=dev).to(torch.bfloat16),
                 torch.randn((100, wl.H, wl.D), generator=g, device=dev).to(torch.bfloat16)) for _ in lengths]
        table = kvq.RequestTable(pool.k_streams, pool.v_streams, dev, segments=tail)
        ws = torch.empty(kvq.kvq_decode_attn_workspace_bytes(len(lengths), wl.H, wl.Hq, wl.D), dtype=torch.uint8,
                         device=dev)
        for _ in range(args.reps):
            kvq.kvq_decode_attn_packed(table, wl.q, wl.depth, wl.H, workspace=ws)
    torch.cuda.synchronize()
    err = kvq.attn_error_word(pool.workspace)
    if args.stage in ("attention", "tail"):
        err |= kvq.attn_error_word(ws)
    elif args.stage == "sparse":
        err |= kvq.attn_error_word(st.workspace) | kvq.attn_error_word(ws)
    print("ok" if err == 0 else f"error word {err}")
    return 0 if err == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
