"""GPU parity of the prefill path through the C ABI: qsa_indexer_prefill and
qsa_sparse_prefill against the fp64 CPU oracle on the same seeded inputs.

Indexer: block keys bit-exact (both sides round an f64 value to fp16), lists
equal as sets except for swaps at the cut within the 1e-6 relative tie band,
and the list contract checked on every row.  Attention: the oracle's own
lists feed both sides; max |gpu - f64| <= 2e-3, exact zeros on padded rows.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_qsa_gb300 import _binding as qb
from block_sparse_gqa_qsa_gb300 import synthetic as syn
from qsa_testlib import (check_attention, check_list, check_lists_device, compare_selection, f32,
                         gpu_indexer_prefill, oracle_prefill_lists, same_fp16_bits, to_np, workspace_kbar)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_gqa_qsa_gb300 import build
    build.build()
    qb.lib()


def _inputs(cfg, poison=True):
    t = syn.make_prefill(cfg, poison=poison)
    t_np = {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    t_dev = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    return t_np, t_dev


def _check_indexer(cfg, t_np, t_dev, rows=None):
    ind, ws = gpu_indexer_prefill(t_dev, cfg)
    torch.cuda.synchronize()
    check_lists_device(ind, t_np["ctx"], cfg.ratio, cfg.budget)
    # block keys: bit-exact
    _, kb_ref = oracle.indexer_prefill(t_np["idxQ"], t_np["idxK"], t_np["wq"], t_np["wk"], t_np["ctx"],
                                       rot=cfg.rot, ratio=cfg.ratio, budget=cfg.budget, topK=cfg.topK,
                                       theta=cfg.theta, eps=f32(cfg.eps), rows=np.zeros(1, np.int64),
                                       want_kbar=True)
    kb_gpu = workspace_kbar(ws, cfg.B, cfg.S, cfg.di, cfg.ratio)
    for b in range(cfg.B):
        nb = int(t_np["ctx"][b]) // cfg.ratio
        assert same_fp16_bits(kb_gpu[b, :nb], kb_ref[b, :nb]), f"block keys of sequence {b} differ"
    # lists: sets with the tie tolerance
    if rows is None:
        rows = np.arange(cfg.B * cfg.S, dtype=np.int64)
    ora, sc = oracle_prefill_lists(t_np, cfg, rows=rows, want_scores=True)
    gpu = to_np(ind).reshape(cfg.B * cfg.S, cfg.topK)[rows]
    equal = 0
    for i, row in enumerate(rows):
        b, t = divmod(int(row), cfg.S)
        L = int(t_np["ctx"][b])
        if t >= L:
            assert np.all(gpu[i] == -1)
            continue
        check_list(gpu[i], t, L, cfg.ratio, cfg.budget)
        equal += compare_selection(gpu[i], ora[i], sc[i], t, cfg.ratio, cfg.budget)
    return ind, equal


@pytest.mark.parametrize("cfg", [syn.PREFILL_TINY, syn.PREFILL_PARITY], ids=lambda c: c.name)
def test_indexer_prefill_parity(cfg):
    t_np, t_dev = _inputs(cfg)
    _check_indexer(cfg, t_np, t_dev)


def test_indexer_prefill_edges():
    base = syn.PREFILL_PARITY
    cases = [
        dataclasses.replace(base, name="dense", B=1, S=700, budget=200, ctx_lo=None, ctx_hi=None),
        dataclasses.replace(base, name="tiny_S3", B=2, S=3, budget=4, ctx_lo=0, ctx_hi=3),
        dataclasses.replace(base, name="odd_S", B=3, S=1029, budget=64, ctx_lo=0, ctx_hi=1029, seed=3),
        dataclasses.replace(base, name="di64_Hi3", B=1, S=1500, Hi=3, di=64, rot=16, budget=100, ctx_lo=None,
                            ctx_hi=None, seed=4),
        dataclasses.replace(base, name="rot_full", B=1, S=900, rot=128, budget=50, ctx_lo=None, ctx_hi=None,
                            seed=5),
        # ratios other than 4 run the top-k instance that reads r from its arguments
        dataclasses.replace(base, name="ratio3", B=1, S=1400, ratio=3, budget=60, ctx_lo=None, ctx_hi=None, seed=6),
        dataclasses.replace(base, name="ratio8", B=2, S=2100, ratio=8, budget=40, ctx_lo=900, ctx_hi=2100, seed=8),
    ]
    for cfg in cases:
        t_np, t_dev = _inputs(cfg)
        _check_indexer(cfg, t_np, t_dev)


def test_indexer_prefill_wider_topk_pads():
    cfg = dataclasses.replace(syn.PREFILL_PARITY, B=1, S=1200, budget=40, ctx_lo=None, ctx_hi=None)
    t_np, t_dev = _inputs(cfg)
    topK = cfg.topK + 29
    ind, _ = gpu_indexer_prefill(t_dev, cfg, topK=topK)
    ora = oracle_prefill_lists(t_np, cfg, topK=topK)
    g, o = to_np(ind), ora
    assert np.all(g[..., cfg.topK:] == -1)
    sc = oracle_prefill_lists(t_np, cfg, want_scores=True, rows=np.arange(cfg.S, dtype=np.int64))[1]
    for t in range(cfg.S):
        compare_selection(g[0, t], o[0, t], sc[t], t, cfg.ratio, cfg.budget)


@pytest.mark.parametrize("S,budget", [(1100, 30), (6000, 300)])
def test_indexer_prefill_exact_ties_take_lowest_ids(S, budget):
    """Identical block keys (no RoPE) tie exactly on both sides; so do all-zero scores.

    At S = 6000 a row's 1500 tied keys exceed what the select stages in shared
    memory, so the cut is narrowed over the scores in global memory first."""
    cfg = dataclasses.replace(syn.PREFILL_PARITY, B=2, S=S, rot=0, budget=budget, ctx_lo=None, ctx_hi=None)
    t_np, t_dev = _inputs(cfg)
    x = t_np["idxK"][0, 0].copy()
    t_np["idxK"][:] = x
    t_np["idxQ"][1] = -x  # sequence 1: every dot negative -> every score exactly 0
    t_dev["idxK"] = torch.from_numpy(t_np["idxK"]).to(DEV)
    t_dev["idxQ"] = torch.from_numpy(t_np["idxQ"]).to(DEV)
    t_np["wq"][:] = 0
    t_np["wk"][:] = 0
    t_dev["wq"].zero_()
    t_dev["wk"].zero_()
    ind, _ = gpu_indexer_prefill(t_dev, cfg)
    ora = oracle_prefill_lists(t_np, cfg)
    assert np.array_equal(to_np(ind), ora)


def test_indexer_prefill_clustered_scores_refine_the_cut():
    """Most blocks score inside a narrow band, seven octaves above a dozen tiny outliers.

    The row's positive keys then span ~2^26 bit patterns while the cut sits
    among hundreds of keys a few thousand patterns apart, so the top-k's radix
    select narrows the cut's bin two or three times before it ranks the last
    few keys (the keys live in the dims past rot, which RoPE leaves alone).
    """
    cfg = dataclasses.replace(syn.PREFILL_PARITY, B=1, S=2000, budget=50, ctx_lo=None, ctx_hi=None, seed=11)
    t_np, t_dev = _inputs(cfg, poison=False)
    rng = np.random.default_rng(11)
    di, rot, r = cfg.di, cfg.rot, cfg.ratio
    m = (np.arange(di) >= rot).astype(np.float32)
    base = m * rng.uniform(0.5, 1.5, di).astype(np.float32)
    u = m * rng.standard_normal(di).astype(np.float32)
    u -= base * (u @ base) / (base @ base)  # orthogonal to the common direction
    K = base[None, :] + 0.02 * rng.standard_normal((cfg.S, di)).astype(np.float32) * m
    for g in rng.choice(cfg.S // r, 12, replace=False):
        K[g * r:(g + 1) * r] = u + 0.001 * base
    Q = base[None, None, :] + 0.05 * rng.standard_normal((cfg.S, cfg.Hi, di)).astype(np.float32) * m
    t_np["idxK"][0] = K.astype(np.float16)
    t_np["idxQ"][0] = Q.astype(np.float16)
    t_dev["idxK"] = torch.from_numpy(t_np["idxK"]).to(DEV)
    t_dev["idxQ"] = torch.from_numpy(t_np["idxQ"]).to(DEV)
    _check_indexer(cfg, t_np, t_dev)


@pytest.mark.parametrize("cfg", [syn.PREFILL_8K, syn.PREFILL_RAGGED], ids=lambda c: c.name)
def test_indexer_prefill_full_size(cfg):
    t_np, t_dev = _inputs(cfg)
    rng = np.random.default_rng(0)
    rows = []
    for b in range(cfg.B):
        L = int(t_np["ctx"][b])
        pick = set(rng.integers(0, L, size=96).tolist()) | {0, 1, 2047, 2048, 2051, L - 2, L - 1}
        pick |= {L, min(cfg.S - 1, L + 5)} if L < cfg.S else set()
        rows += [b * cfg.S + r for r in sorted(pick) if 0 <= r < cfg.S]
    _check_indexer(cfg, t_np, t_dev, rows=np.array(rows, np.int64))


@pytest.mark.parametrize("cfg", [syn.PREFILL_28K, syn.PREFILL_64K, syn.PREFILL_LONG_RAGGED],
                         ids=lambda c: c.name)
def test_indexer_prefill_long(cfg):
    """Sequences past 16K rows: every list's structure on the device, block keys
    bit-exact, and sampled rows (random, around the budget and at the ends)
    against the oracle's selection.  At 64K the longest rows hold more keys in
    the cut's histogram bin than the select stages in shared memory."""
    t_np, t_dev = _inputs(cfg)
    rng = np.random.default_rng(cfg.seed)
    rows = []
    for b in range(cfg.B):
        L = int(t_np["ctx"][b])
        pick = set(rng.integers(0, L, size=40).tolist()) | {0, 2050, 2051, 16383, 16387, L - 2, L - 1}
        pick |= set(rng.integers(max(0, L - 2000), L, size=16).tolist())
        pick |= {L, min(cfg.S - 1, L + 5)} if L < cfg.S else set()
        rows += [b * cfg.S + r for r in sorted(pick) if 0 <= r < cfg.S]
    _check_indexer(cfg, t_np, t_dev, rows=np.array(rows, np.int64))


def test_indexer_prefill_workspace_reuse_across_shapes():
    """One workspace serves a long call, then a short one, then the long one
    again: the work counter is re-armed by every call and no score slot
    carries state from one call to the next."""
    long_cfg = dataclasses.replace(syn.PREFILL_LONG_RAGGED, B=1, S=18000, ctx_lo=None, ctx_hi=None, seed=21)
    short_cfg = syn.PREFILL_PARITY
    tl_np, tl = _inputs(long_cfg)
    ts_np, ts = _inputs(short_cfg)
    ws = qb.alloc_workspace(qb.indexer_prefill_workspace_size(1, long_cfg.S, long_cfg.di, long_cfg.ratio), DEV)
    outs = []
    for cfg, t in ((long_cfg, tl), (short_cfg, ts), (long_cfg, tl)):
        ind = torch.full((cfg.B, cfg.S, cfg.topK), 7, dtype=torch.int32, device=DEV)
        qb.indexer_prefill(t["idxQ"], t["idxK"], t["wq"], t["wk"], t["ctx"], ind, ws, rot=cfg.rot, ratio=cfg.ratio,
                           budget=cfg.budget, topK=cfg.topK, theta=cfg.theta, eps=cfg.eps)
        outs.append(ind)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[2])
    ref, _ = gpu_indexer_prefill(ts, short_cfg)
    assert torch.equal(outs[1], ref)
    check_lists_device(outs[0], tl_np["ctx"], long_cfg.ratio, long_cfg.budget)


# ------------------------------------------------------------------ attention
IMPLS = ("mma", "tcgen05")  # mma.sync tiles, and the tcgen05 / TMEM variant of the same contract


def _gpu_attention(t_dev, lists_dev, cfg, scale, impl="mma"):
    out = torch.full((cfg.B, cfg.S, cfg.Hq, cfg.D), float("nan"), dtype=torch.float16, device=DEV)
    qb.sparse_prefill(t_dev["q"], t_dev["k"], t_dev["v"], lists_dev, t_dev["ctx"], out, scale, impl=impl)
    torch.cuda.synchronize()
    return out


def _check_rows(out, t_np, lists_np, cfg, rows, scale, what):
    ref = oracle.sparse_prefill(t_np["q"], t_np["k"], t_np["v"], lists_np.reshape(-1, lists_np.shape[-1])[rows],
                                t_np["ctx"], scale, rows=rows)
    got = to_np(out).reshape(-1, cfg.Hq, cfg.D)[rows]
    err = check_attention(got, ref, what)
    for i, row in enumerate(rows):  # padded rows: exact fp16 zeros
        b, t = divmod(int(row), cfg.S)
        if t >= int(t_np["ctx"][b]):
            assert np.all(got[i].view(np.uint16) == 0), f"{what}: padded row {t} not exactly zero"
    return err


@pytest.mark.parametrize("impl", IMPLS)
def test_sparse_prefill_status_word_reports_bad_entries(impl):
    """Entries past the live length or negative (other than the -1 padding)
    are skipped without a fault, and the optional status word's bit 2 says so;
    the output equals the oracle's on the lists with those entries dropped."""
    cfg = dataclasses.replace(syn.PREFILL_PARITY, B=2, S=900, ctx_lo=500, ctx_hi=900, seed=31)
    t_np, t_dev = _inputs(cfg)
    lists = oracle_prefill_lists(t_np, cfg)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty((cfg.B, cfg.S, cfg.Hq, cfg.D), dtype=torch.float16, device=DEV)
    qb.sparse_prefill(t_dev["q"], t_dev["k"], t_dev["v"], torch.from_numpy(lists).to(DEV), t_dev["ctx"], out,
                      f32(cfg.scale), status=status, impl=impl)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "clean lists set a status bit"
    bad = lists.copy()
    L0 = int(t_np["ctx"][0])
    bad[0, 400, 3] = L0 + 7         # past the live length
    bad[0, 401, 0] = -9             # negative, not the padding
    bad[1, 10, 2] = 1 << 30         # far out of range
    want = lists.copy()
    want[0, 400, 3] = want[0, 401, 0] = want[1, 10, 2] = -1
    out = _gpu_attention(t_dev, torch.from_numpy(bad).to(DEV), cfg, f32(cfg.scale), impl)
    qb.sparse_prefill(t_dev["q"], t_dev["k"], t_dev["v"], torch.from_numpy(bad).to(DEV), t_dev["ctx"], out,
                      f32(cfg.scale), status=status, impl=impl)
    torch.cuda.synchronize()
    assert int(status.item()) == 4, f"status {int(status.item())} != bit 2"
    rows = np.array([400, 401, 402, cfg.S + 10, cfg.S + 11], np.int64)
    _check_rows(out, t_np, want, cfg, rows, f32(cfg.scale), "bad entries dropped")


@pytest.mark.parametrize("impl", IMPLS)
def test_sparse_prefill_parity_oracle_lists(impl):
    cfg = syn.PREFILL_PARITY
    t_np, t_dev = _inputs(cfg)
    lists = oracle_prefill_lists(t_np, cfg)
    out = _gpu_attention(t_dev, torch.from_numpy(lists).to(DEV), cfg, f32(cfg.scale), impl)
    rows = np.arange(cfg.B * cfg.S, dtype=np.int64)
    _check_rows(out, t_np, lists, cfg, rows, f32(cfg.scale), "parity")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (16, 2), (32, 2), (24, 2)])
def test_sparse_prefill_group_sizes_and_list_shapes(Hq, Hkv, impl):
    cfg = dataclasses.replace(syn.PREFILL_PARITY, name=f"g{Hq // Hkv}", B=2, S=700, Hq=Hq, Hkv=Hkv,
                              ctx_lo=300, ctx_hi=700, seed=Hq)
    t_np, t_dev = _inputs(cfg)
    rows = np.arange(cfg.B * cfg.S, dtype=np.int64)
    # random order, causal
    lists = syn.random_lists(cfg.B, cfg.S, 150, t_np["ctx"], seed=1, fill=0.7).numpy()
    out = _gpu_attention(t_dev, torch.from_numpy(lists).to(DEV), cfg, 0.07, impl)
    _check_rows(out, t_np, lists, cfg, rows, f32(0.07), "random causal")
    # non-causal entries (no positional mask), several tiles wide
    lists = syn.random_lists(cfg.B, cfg.S, 300, t_np["ctx"], seed=2, fill=0.9, causal=False).numpy()
    out = _gpu_attention(t_dev, torch.from_numpy(lists).to(DEV), cfg, 0.1, impl)
    _check_rows(out, t_np, lists, cfg, rows, f32(0.1), "non-causal")


def test_prefill_many_sequences():
    """Forty sequences of random length up to 1100, four of them 0, 1, 3 and 4 tokens long: the indexer's
    work items cycle over every sequence (lists checked on every row) and both attention kernels run the
    indexer's own lists (checked on every seventh row)."""
    cfg = dataclasses.replace(syn.PREFILL_PARITY, name="many_seqs", B=40, S=1100, budget=64, ctx_lo=0,
                              ctx_hi=1100, seed=9)
    t_np, t_dev = _inputs(cfg)
    t_np["ctx"][:4] = (0, 1, 3, 4)  # rows past these lengths keep data: they are never read either way
    t_dev["ctx"] = torch.from_numpy(t_np["ctx"]).to(DEV)
    ind, _ = _check_indexer(cfg, t_np, t_dev)
    lists = to_np(ind)
    rows = np.arange(0, cfg.B * cfg.S, 7, dtype=np.int64)
    for impl in IMPLS:
        out = _gpu_attention(t_dev, ind, cfg, f32(cfg.scale), impl)
        _check_rows(out, t_np, lists, cfg, rows, f32(cfg.scale), f"many sequences ({impl})")


@pytest.mark.parametrize("impl", IMPLS)
def test_sparse_prefill_special_lists(impl):
    cfg = dataclasses.replace(syn.PREFILL_PARITY, B=1, S=300, ctx_lo=None, ctx_hi=None)
    t_np, t_dev = _inputs(cfg)
    topK = 67
    rng = np.random.default_rng(5)
    lists = np.full((1, cfg.S, topK), -1, np.int32)
    js = rng.integers(0, cfg.S, size=cfg.S)
    lists[0, :, 0] = js  # one entry: the output is that value row, exactly
    lists[0, 7] = -1     # empty list: zeros
    out = to_np(_gpu_attention(t_dev, torch.from_numpy(lists).to(DEV), cfg, 0.09, impl))
    for t in range(cfg.S):
        for h in range(cfg.Hq):
            want = np.zeros(cfg.D, np.float16) if t == 7 else t_np["v"][0, js[t], h // (cfg.Hq // cfg.Hkv)]
            assert np.array_equal(out[0, t, h].view(np.uint16), want.view(np.uint16)), (t, h)
    # entries at or past L are skipped, as if absent
    cfg2 = dataclasses.replace(cfg, ctx_lo=200, ctx_hi=200)
    t_np, t_dev = _inputs(cfg2)
    lists = syn.random_lists(1, cfg.S, topK, t_np["ctx"], seed=3, fill=0.5).numpy()
    bad = lists.copy()
    bad[0, :200, -1] = 250  # names a padded (NaN) row
    out = _gpu_attention(t_dev, torch.from_numpy(bad).to(DEV), cfg2, 0.09, impl)
    _check_rows(out, t_np, lists, cfg2, np.arange(cfg.S, dtype=np.int64), f32(0.09), "skip >= L")


@pytest.mark.parametrize("impl", IMPLS)
def test_sparse_prefill_full_size_8k(impl):
    cfg = syn.PREFILL_8K
    t_np, t_dev = _inputs(cfg)
    lists = oracle_prefill_lists(t_np, cfg)
    out = _gpu_attention(t_dev, torch.from_numpy(lists).to(DEV), cfg, f32(cfg.scale), impl)
    rows = np.unique(np.concatenate([np.arange(0, 8192, 97), [1, 2047, 2048, 2049, 8190, 8191]])).astype(np.int64)
    _check_rows(out, t_np, lists, cfg, rows, f32(cfg.scale), "8k")
    assert not torch.isnan(out).any()


@pytest.mark.parametrize("impl", IMPLS)
def test_sparse_prefill_full_size_ragged(impl):
    cfg = syn.PREFILL_RAGGED
    t_np, t_dev = _inputs(cfg)
    lists_dev = syn.qsa_like_lists(cfg.B, cfg.S, t_np["ctx"], cfg.ratio, cfg.budget, cfg.topK, seed=9, device=DEV)
    out = _gpu_attention(t_dev, lists_dev, cfg, f32(cfg.scale), impl)
    lists = to_np(lists_dev)
    rows = []
    for b in range(cfg.B):
        L = int(t_np["ctx"][b])
        rows += [b * cfg.S + r for r in (0, 5, L // 2, L - 1, L, cfg.S - 1) if r < cfg.S]
        rows += [b * cfg.S + r for r in range(0, cfg.S, 997)]
    rows = np.unique(np.array(rows, np.int64))
    _check_rows(out, t_np, lists, cfg, rows, f32(cfg.scale), "ragged")
    for b in range(cfg.B):  # every padded row of every sequence is exactly zero
        L = int(t_np["ctx"][b])
        assert bool((out[b, L:].view(torch.int16) == 0).all())
    assert not torch.isnan(out).any()


@pytest.mark.parametrize("impl", IMPLS)
def test_prefill_end_to_end_8k(impl):
    """Raw inputs through both whole paths; sets agree up to ties, outputs agree where sets do."""
    cfg = syn.PREFILL_8K
    t_np, t_dev = _inputs(cfg)
    ind, _ = gpu_indexer_prefill(t_dev, cfg)
    out = _gpu_attention(t_dev, ind, cfg, f32(cfg.scale), impl)
    rows = np.arange(0, cfg.S, 61, dtype=np.int64)
    ora, sc = oracle_prefill_lists(t_np, cfg, rows=rows, want_scores=True)
    gpu = to_np(ind)[0][rows]
    same = [i for i, r in enumerate(rows) if compare_selection(gpu[i], ora[i], sc[i], int(r), cfg.ratio, cfg.budget)]
    assert len(same) >= 0.95 * len(rows)
    ref = oracle.sparse_prefill(t_np["q"], t_np["k"], t_np["v"], ora[same], t_np["ctx"], f32(cfg.scale),
                                rows=rows[same])
    check_attention(to_np(out)[0][rows[same]], ref, "end-to-end")
