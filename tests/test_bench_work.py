"""The work counts behind the bench's roofline lines, checked on CPU against
independent counts: the entries of the oracle's own index lists (the gathered
rows of the attention), and a row-by-row loop over the scoring rule (the
indexer's block-score FMAs)."""
from __future__ import annotations

import dataclasses

import numpy as np

import bench
from block_sparse_gqa_qsa_gb300 import synthetic as syn
from qsa_testlib import oracle_prefill_lists


def _ragged_tiny():
    # two sequences of different live length, both past the budget (n_c > 16), one of them padded
    return dataclasses.replace(syn.PREFILL_TINY, name="tiny_ragged", B=2, ctx_lo=300, ctx_hi=512, seed=1201)


def test_prefill_work_matches_the_oracle_lists():
    for cfg in (syn.PREFILL_TINY, _ragged_tiny()):
        t = syn.make_prefill(cfg)
        t_np = {k: v.numpy() for k, v in t.items()}
        ctx = [int(x) for x in t_np["ctx"]]
        lists = oracle_prefill_lists(t_np, cfg).reshape(cfg.B, cfg.S, cfg.topK)
        live = sum(int(np.sum(lists[b, :L] >= 0)) for b, L in enumerate(ctx))
        assert all(np.all(lists[b, L:] == -1) for b, L in enumerate(ctx))
        tok, cnt, gbytes, flops = bench.prefill_work(cfg, ctx)
        assert tok == sum(ctx)
        assert cnt == live, f"{cfg.name}: {cnt} list entries counted, the oracle's lists hold {live}"
        # every live entry is one K row and one V row per KV head; Q read and O written once per live row
        assert gbytes == cfg.Hkv * live * 2 * cfg.D * 2 + 2 * sum(ctx) * cfg.Hq * cfg.D * 2 + \
            cfg.B * cfg.S * cfg.topK * 4
        # S = q.k and O += p.v: two multiply-adds per entry, head and dim
        assert flops == 2 * 2 * live * cfg.Hq * cfg.D


def test_indexer_fma_counts_the_scored_rows():
    cfg = _ragged_tiny()
    ctx = [int(x) for x in syn.context_lengths(cfg)]
    want = 0
    for L in ctx:
        for t in range(L):
            n_c = (t + 1) // cfg.ratio
            if n_c > cfg.budget:  # rows at or under the budget keep every block without scoring
                want += n_c * cfg.Hi * cfg.di
    assert bench.indexer_fma(cfg, ctx) == want


def test_decode_work_matches_the_oracle_lists():
    import oracle
    from qsa_testlib import f32
    cfg = syn.DECODE_PARITY
    d = syn.make_decode(cfg)
    d_np = {k: (v.numpy() if hasattr(v, "numpy") else v) for k, v in d.items()}
    ctx = [int(x) for x in d_np["ctx"]]
    lists = oracle.indexer_decode(d_np["idxQ"], d_np["idxK"], d_np["wq"], d_np["wk"], d_np["pool"].copy(),
                                  d_np["page_table"], d_np["ctx"], D=cfg.D, rot=cfg.rot, ratio=cfg.ratio,
                                  budget=cfg.budget, topK=cfg.topK, theta=cfg.theta, eps=f32(cfg.eps))
    live = int(np.sum(lists >= 0))
    kbar, kv, total = bench.decode_work(cfg, ctx)
    # the scorer streams one key per complete block of the new token's row t = L - 1
    assert kbar == sum((L // cfg.ratio) * cfg.di * 2 for L in ctx)
    assert kv == cfg.Hkv * live * 2 * cfg.D * 2, "gathered rows must be the oracle lists' entries"
    assert total == kbar + kv + cfg.B * (2 * cfg.Hq * cfg.D * 2 + cfg.Hi * cfg.di * 2 + cfg.topK * 4 * 2)


def test_end_to_end_copies_cover_exactly_the_live_rows():
    import torch
    cfg = _ragged_tiny()
    t = syn.make_prefill(cfg)  # rows at or past each length are NaN
    ctx = [int(x) for x in t["ctx"]]
    dst = {k: torch.full_like(v, -7) for k, v in t.items()}
    pairs = [p for k in t for p in bench.live_copies(cfg, ctx, dst[k], t[k])]
    for d, s_ in pairs:
        assert d.is_contiguous() and s_.is_contiguous()
        d.copy_(s_)
    want = sum(v.numel() * v.element_size() for k, v in t.items() if k in ("wq", "wk", "ctx"))
    for k in ("q", "k", "v", "idxQ", "idxK"):
        row = t[k][0, 0].numel() * t[k].element_size()
        want += sum(ctx) * row
        for b, L in enumerate(ctx):
            assert torch.equal(dst[k][b, :L], t[k][b, :L]), f"{k}: live rows of sequence {b} not copied"
            assert torch.all(dst[k][b, L:] == -7), f"{k}: padded rows of sequence {b} were copied"
    assert sum(s_.numel() * s_.element_size() for _, s_ in pairs) == want
    for k in ("wq", "wk", "ctx"):
        assert torch.equal(dst[k], t[k])
