"""Runs a few steps of one named workload on cuda:0 through the C ABI.

A step is the whole path for that workload: qsa_indexer_prefill +
qsa_sparse_prefill for a prefill workload, qsa_indexer_decode +
qsa_sparse_decode for a decode workload.  Inputs come from the seeded
generators of `synthetic`.  The sizes can be overridden to get a case small
enough for a profiler's multi-pass capture (a decode pool of a few GB instead
of tens).

    python -m block_sparse_gqa_qsa_gb300.run_case prefill_S8192 --steps 2
    python -m block_sparse_gqa_qsa_gb300.run_case decode_long_B8_L512k --B 1 --steps 2
    python -m block_sparse_gqa_qsa_gb300.run_case prefill_S8192 --op rope --steps 2
    python -m block_sparse_gqa_qsa_gb300.run_case prefill_S8192 --impl tcgen05 --steps 1

`--op rope` runs qsa_rope_qkv on the workload's packed QKV instead (prefill
workloads: dense q/k/v outputs).  `--op handoff` (prefill workloads) runs the
indexer once, then qsa_indexer_prefill_handoff into a paged pool per step.
`--op gather` (decode workloads) runs one decode step for its lists, then
qsa_gather_selected into contiguous scratch per step.
"""
from __future__ import annotations

import argparse
import dataclasses
import math

import torch

from . import _binding as qb
from . import synthetic as syn


def _prefill_steps(cfg, steps, impl="mma"):
    t = {k: v.cuda() for k, v in syn.make_prefill(cfg).items()}
    ws = qb.alloc_workspace(qb.indexer_prefill_workspace_size(cfg.B, cfg.S, cfg.di, cfg.ratio))
    ind = torch.empty((cfg.B, cfg.S, cfg.topK), dtype=torch.int32, device="cuda")
    out = torch.empty((cfg.B, cfg.S, cfg.Hq, cfg.D), dtype=torch.float16, device="cuda")
    scale = float(torch.tensor(1.0 / math.sqrt(cfg.D), dtype=torch.float32))
    for _ in range(steps):
        qb.indexer_prefill(t["idxQ"], t["idxK"], t["wq"], t["wk"], t["ctx"], ind, ws, rot=cfg.rot, ratio=cfg.ratio,
                           budget=cfg.budget, topK=cfg.topK, theta=cfg.theta, eps=cfg.eps)
        qb.sparse_prefill(t["q"], t["k"], t["v"], ind, t["ctx"], out, scale, impl=impl)


def _rope_steps(cfg, steps):
    t = syn.make_prefill(cfg)
    qkv = torch.cat([t["q"], t["k"], t["v"]], dim=2).contiguous().cuda()
    wq, wk, ctx = t["wq"].cuda(), t["wk"].cuda(), t["ctx"].cuda()
    qo = torch.empty((cfg.B, cfg.S, cfg.Hq, cfg.D), dtype=torch.float16, device="cuda")
    ko = torch.empty((cfg.B, cfg.S, cfg.Hkv, cfg.D), dtype=torch.float16, device="cuda")
    vo = torch.empty_like(ko)
    for _ in range(steps):
        qb.rope_qkv(qkv, wq, wk, ctx, qo, Hq=cfg.Hq, Hkv=cfg.Hkv, rot=cfg.rot, theta=cfg.theta, eps=cfg.eps,
                    k_out=ko, v_out=vo)


def _handoff_steps(cfg, steps):
    t = {k: v.cuda() for k, v in syn.make_prefill(cfg).items()}
    ws = qb.alloc_workspace(qb.indexer_prefill_workspace_size(cfg.B, cfg.S, cfg.di, cfg.ratio))
    ind = torch.empty((cfg.B, cfg.S, cfg.topK), dtype=torch.int32, device="cuda")
    qb.indexer_prefill(t["idxQ"], t["idxK"], t["wq"], t["wk"], t["ctx"], ind, ws, rot=cfg.rot, ratio=cfg.ratio,
                       budget=cfg.budget, topK=cfg.topK, theta=cfg.theta, eps=cfg.eps)
    npg = -(-(cfg.S + 1) // syn.TOKENS_PER_PAGE)  # pages for S tokens and the next one, per sequence
    pool = torch.zeros((2 * cfg.B * npg, syn.TOKENS_PER_PAGE, cfg.Hkv, cfg.D + cfg.di), dtype=torch.float16,
                       device="cuda")
    ids = torch.arange(cfg.B * npg, dtype=torch.int32, device="cuda").view(cfg.B, npg)
    pt = torch.stack([ids, ids + cfg.B * npg], dim=1).contiguous()
    for _ in range(steps):
        qb.indexer_prefill_handoff(t["idxK"], t["ctx"], ws, pool, pt, D=cfg.D, ratio=cfg.ratio)


def _gather_steps(cfg, steps):
    d, ind = _decode_steps(cfg, 1)
    sc = qb.gather_scratch(cfg.B, cfg.Hkv, cfg.D, cfg.topK, device="cuda")
    for _ in range(steps):
        qb.gather_selected(d["pool"], d["page_table"], ind, d["ctx"], *sc, D=cfg.D)


def _decode_steps(cfg, steps):
    d = syn.make_decode(cfg, device="cuda")
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    ws = qb.alloc_workspace(qb.indexer_decode_workspace_size(cfg.B, cfg.maxPagesPerSeq, cfg.ratio, cfg.budget))
    po, ps, pc = qb.sparse_decode_workspace_elems(cfg.B, cfg.Hkv, cfg.D)
    parts = (torch.zeros(po, device="cuda"), torch.zeros(ps, device="cuda"),
             torch.zeros(pc, dtype=torch.int32, device="cuda"))
    ind = torch.empty((cfg.B, 1, cfg.topK), dtype=torch.int32, device="cuda")
    out = torch.empty((cfg.B, 1, cfg.Hq, cfg.D), dtype=torch.float16, device="cuda")
    scale = float(torch.tensor(1.0 / math.sqrt(cfg.D), dtype=torch.float32))
    for _ in range(steps):
        qb.indexer_decode(d["idxQ"], d["idxK"], d["wq"], d["wk"], d["pool"], d["page_table"], d["ctx"], ind, ws,
                          D=cfg.D, rot=cfg.rot, ratio=cfg.ratio, budget=cfg.budget, topK=cfg.topK, theta=cfg.theta,
                          eps=cfg.eps)
        qb.sparse_decode(d["q"], d["pool"], d["page_table"], ind, d["ctx"], out, *parts, D=cfg.D, scale=scale)
    return d, ind


def main(argv=None):
    names = {c.name: c for c in syn.BENCH_CONFIGS + (syn.PREFILL_28K, syn.PREFILL_64K)}
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("workload", choices=sorted(names))
    ap.add_argument("--steps", type=int, default=2)
    ap.add_argument("--B", type=int, default=None, help="override the batch size")
    ap.add_argument("--ctx", type=int, default=None, help="decode: every sequence gets this total length")
    ap.add_argument("--Hkv", type=int, default=None,
                    help="decode: KV heads of the pool (Hq becomes 8 * Hkv); fewer heads make the pool smaller with "
                         "the same block-key stream per sequence")
    ap.add_argument("--impl", choices=("mma", "tcgen05"), default="mma",
                    help="prefill attention: qsa_sparse_prefill (mma.sync) or qsa_sparse_prefill_tcgen05")
    ap.add_argument("--op", choices=("path", "rope", "handoff", "gather"), default="path",
                    help="rope / handoff: qsa_rope_qkv / qsa_indexer_prefill_handoff of a prefill workload; "
                         "gather: qsa_gather_selected of a decode workload")
    args = ap.parse_args(argv)
    cfg = names[args.workload]
    if args.B is not None:
        cfg = dataclasses.replace(cfg, B=args.B)
    qb.lib()
    if args.op in ("rope", "handoff"):
        if isinstance(cfg, syn.DecodeConfig):
            ap.error(f"--op {args.op} takes a prefill workload")
        (_rope_steps if args.op == "rope" else _handoff_steps)(cfg, args.steps)
    elif args.op == "gather":
        if not isinstance(cfg, syn.DecodeConfig):
            ap.error("--op gather takes a decode workload")
        _gather_steps(cfg, args.steps)
    elif isinstance(cfg, syn.DecodeConfig):
        if args.ctx is not None:
            cfg = dataclasses.replace(cfg, ctx_lo=args.ctx, ctx_hi=args.ctx, max_ctx=max(args.ctx, 1), ctx_list=None)
        if args.Hkv is not None:
            cfg = dataclasses.replace(cfg, Hkv=args.Hkv, Hq=8 * args.Hkv)
        _decode_steps(cfg, args.steps)
    else:
        _prefill_steps(cfg, args.steps, args.impl)
    torch.cuda.synchronize()
    print(f"ok: {args.steps} steps of {cfg.name} (B={cfg.B})")


if __name__ == "__main__":
    main()
