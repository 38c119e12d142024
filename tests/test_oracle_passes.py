"""Pins of the oracle's whole passes (prefill indexer, attention, decode).

Attention is pinned to torch's scaled_dot_product_attention in f64 (the dense
special case), to closed forms (one index -> that value row) and invariances;
the indexer passes to their own step functions' definitions through planted
structure (identical keys, aligned keys) and to the list invariants; the
decode passes to the prefill passes on the same logical data laid out in a
shuffled paged pool.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from block_sparse_gqa_qsa_gb300 import synthetic as syn

TPP = syn.TOKENS_PER_PAGE


def _small_prefill(B=2, S=300, Hq=4, Hkv=2, D=128, Hi=4, di=64, rot=32, ratio=4, budget=8, seed=5,
                   ctx=None):
    cfg = syn.PrefillConfig("t", B=B, S=S, Hq=Hq, Hkv=Hkv, D=D, Hi=Hi, di=di, rot=rot, ratio=ratio,
                            budget=budget, seed=seed)
    t = syn.make_prefill(cfg, poison=False)
    if ctx is not None:
        t["ctx"] = torch.tensor(ctx, dtype=torch.int32)
        for b, L in enumerate(ctx):
            for name in ("q", "k", "v", "idxQ", "idxK"):
                t[name][b, L:] = float("nan")
    return cfg, {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in t.items()}


def _idx(oracle_mod, cfg, t, **kw):
    return oracle_mod.indexer_prefill(t["idxQ"], t["idxK"], t["wq"], t["wk"], t["ctx"], rot=cfg.rot,
                                      ratio=cfg.ratio, budget=cfg.budget, topK=cfg.topK, theta=cfg.theta,
                                      eps=cfg.eps, **kw)


def check_list_invariants(lst, t, L, ratio, budget):
    """Index-list contract: distinct, 0 <= j <= t, -1 only on the right, count = cnt(t)."""
    if t >= L:
        assert np.all(lst == -1)
        return
    n = int(np.sum(lst >= 0))
    assert np.all(lst[:n] >= 0) and np.all(lst[n:] == -1)
    v = lst[:n]
    assert len(np.unique(v)) == n
    assert v.min() >= 0 and v.max() <= t
    n_c = (t + 1) // ratio
    assert n == min(n_c, budget) * ratio + (t + 1 - n_c * ratio)
    # whole blocks plus the whole tail
    tail = set(range(n_c * ratio, t + 1))
    assert tail <= set(v.tolist())
    blocks = {j // ratio for j in v.tolist() if j < n_c * ratio}
    assert {g * ratio + j for g in blocks for j in range(ratio)} | tail == set(v.tolist())


# ----------------------------------------------------------- prefill indexer
def test_indexer_invariants_and_padding_rows(oracle_mod):
    cfg, t = _small_prefill(ctx=[300, 173])
    ind = _idx(oracle_mod, cfg, t)
    for b in range(cfg.B):
        for r in range(cfg.S):
            check_list_invariants(ind[b, r], r, int(t["ctx"][b]), cfg.ratio, cfg.budget)


def test_indexer_dense_special_case(oracle_mod):
    cfg, t = _small_prefill(S=120, budget=40)  # budget >= ceil(S/r): every block kept
    ind = _idx(oracle_mod, cfg, t)
    for r in range(cfg.S):
        assert list(ind[0, r][ind[0, r] >= 0]) == list(range(r + 1))


def test_indexer_identical_keys_tie_to_lowest_ids(oracle_mod):
    cfg, t = _small_prefill(B=1, S=200, rot=0, budget=5)
    t["idxK"][:] = t["idxK"][0, 0]  # every raw key equal; no RoPE -> every block key equal
    ind, sc = _idx(oracle_mod, cfg, t, want_scores=True)
    for r in range(cfg.S):
        n_c = (r + 1) // 4
        assert np.all(sc[r, :n_c] == sc[r, 0])
        if n_c > cfg.budget:
            assert list(ind[0, r][: cfg.budget * 4]) == list(range(cfg.budget * 4))


def test_indexer_planted_aligned_block_is_selected(oracle_mod):
    """A block whose key equals every query (no RoPE) wins: Cauchy-Schwarz."""
    cfg, t = _small_prefill(B=1, S=256, rot=0, budget=4)
    x = t["idxQ"][0, 0, 0].copy()
    t["idxQ"][0, :, :, :] = x
    g_star = 17
    t["idxK"][0, 4 * g_star:4 * g_star + 4] = x
    t["wq"][:] = 0
    t["wk"][:] = 0
    ind = _idx(oracle_mod, cfg, t)
    for r in range(4 * g_star + 3, cfg.S):
        assert set(range(4 * g_star, 4 * g_star + 4)) <= set(ind[0, r].tolist())


def test_indexer_wiring_matches_step_functions(oracle_mod):
    cfg, t = _small_prefill(ctx=[300, 250])
    rows = np.array([0, 3, 35, 299, 300 + 37, 300 + 249], np.int64)
    ind, kbar, sc = _idx(oracle_mod, cfg, t, rows=rows, want_kbar=True, want_scores=True)
    for i, row in enumerate(rows):
        b, r = divmod(int(row), cfg.S)
        # block keys: rows 4g..4g+3 at position 4g
        for g in ((r + 1) // 4 - 1, 0):
            if g < 0:
                continue
            kb, _ = oracle_mod.block_key(t["idxK"][b, 4 * g:4 * g + 4], t["wk"], cfg.rot, 4 * g, cfg.theta,
                                         cfg.eps)
            assert np.array_equal(kb.view(np.uint16), kbar[b, g].view(np.uint16))
        q = np.stack([oracle_mod.index_q(t["idxQ"][b, r, h], t["wq"], cfg.rot, r, cfg.theta, cfg.eps)
                      for h in range(cfg.Hi)])
        n_c = (r + 1) // 4
        for g in range(n_c):
            assert sc[i, g] == oracle_mod.block_score(q, kbar[b, g])
        assert np.all(np.isneginf(sc[i, n_c:]))
        sel = oracle_mod.select(sc[i, :n_c], cfg.budget)
        assert np.array_equal(ind[i], oracle_mod.expand(sel, n_c, r, 4, cfg.topK))


# ---------------------------------------------------------------- attention
def test_attention_dense_case_equals_sdpa(oracle_mod):
    cfg, t = _small_prefill(B=2, S=96, Hq=8, Hkv=2, budget=64, ctx=[96, 61])
    ind = _idx(oracle_mod, cfg, t)
    out = oracle_mod.sparse_prefill(t["q"], t["k"], t["v"], ind, t["ctx"], cfg.scale)
    for b in range(cfg.B):
        L = int(t["ctx"][b])
        q = torch.from_numpy(t["q"][b, :L].astype(np.float64)).transpose(0, 1)  # [Hq, L, D]
        k = torch.from_numpy(t["k"][b, :L].astype(np.float64)).transpose(0, 1)
        v = torch.from_numpy(t["v"][b, :L].astype(np.float64)).transpose(0, 1)
        k = k.repeat_interleave(cfg.Hq // cfg.Hkv, dim=0)
        v = v.repeat_interleave(cfg.Hq // cfg.Hkv, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=cfg.scale)
        np.testing.assert_allclose(out[b, :L], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
        assert np.all(out[b, L:] == 0.0)


def test_attention_single_index_is_value_row(oracle_mod):
    cfg, t = _small_prefill(B=1, S=64, Hq=4, Hkv=2)
    ind = np.full((1, 64, 5), -1, np.int32)
    rng = np.random.default_rng(1)
    js = rng.integers(0, 64, size=64)
    ind[0, :, 0] = js  # non-causal entries included: no positional mask
    out = oracle_mod.sparse_prefill(t["q"], t["k"], t["v"], ind, t["ctx"], cfg.scale)
    for r in range(64):
        for h in range(4):
            np.testing.assert_array_equal(out[0, r, h], t["v"][0, js[r], h // 2].astype(np.float64))


def test_attention_permutation_and_gqa_map(oracle_mod):
    cfg, t = _small_prefill(B=1, S=80, Hq=6, Hkv=3)
    lists = syn.random_lists(1, 80, 40, t["ctx"], seed=3, fill=0.8).numpy()
    out = oracle_mod.sparse_prefill(t["q"], t["k"], t["v"], lists, t["ctx"], cfg.scale)
    rng = np.random.default_rng(2)
    shuf = lists.copy()
    for r in range(80):
        n = int(np.sum(lists[0, r] >= 0))
        shuf[0, r, :n] = rng.permutation(lists[0, r, :n])
    out2 = oracle_mod.sparse_prefill(t["q"], t["k"], t["v"], shuf, t["ctx"], cfg.scale)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-13)
    # GQA: heads 2h, 2h+1 read KV head h; a constant V head shows up only there
    v = t["v"].copy()
    v[0, :, 1, :] = 3.0
    out3 = oracle_mod.sparse_prefill(t["q"], t["k"], v, lists, t["ctx"], cfg.scale)
    np.testing.assert_allclose(out3[0, :, 2:4], 3.0, rtol=1e-14)
    for h in (0, 1, 4, 5):
        np.testing.assert_array_equal(out3[0, :, h], out[0, :, h])


def test_attention_empty_list_scale_and_padding(oracle_mod):
    cfg, t = _small_prefill(B=1, S=40, Hq=2, Hkv=1, ctx=[30])
    lists = syn.random_lists(1, 40, 20, t["ctx"], seed=4).numpy()
    lists[0, 5] = -1  # an empty list on a live row -> zeros
    out = oracle_mod.sparse_prefill(t["q"], t["k"], t["v"], lists, t["ctx"], 0.125)
    assert np.all(out[0, 5] == 0) and np.all(out[0, 30:] == 0)
    q2 = (t["q"].astype(np.float32) * 2).astype(np.float16)  # exact doubling in fp16
    out2 = oracle_mod.sparse_prefill(q2, t["k"], t["v"], lists, t["ctx"], 0.0625)
    np.testing.assert_allclose(out2[0, :30], out[0, :30], rtol=0, atol=1e-13)
    bad = lists.copy()
    bad[0, 3, 0] = 35  # names a padded row
    with pytest.raises(ValueError):
        oracle_mod.sparse_prefill(t["q"], t["k"], t["v"], bad, t["ctx"], 0.125)


# ------------------------------------------------------------------- decode
def _pool_from_dense(idxK_dense, k_dense, v_dense, L_list, Hkv, D, di, maxPages, seed, fill_tails=True):
    """Lay dense per-sequence data into a paged pool with shuffled pages.

    K-row tails hold raw index keys of every token, V-row tails of tokens 4g hold
    NaN except where the caller writes block keys; V pages = K pages + numPages."""
    rng = np.random.default_rng(seed)
    B = len(L_list)
    pages = [-(-L // TPP) for L in L_list]
    numPages = sum(pages)
    perm = rng.permutation(numPages)
    pool = np.full((2 * numPages, TPP, Hkv, D + di), np.nan, np.float16)
    pt = np.zeros((B, 2, maxPages), np.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, 0, :n] = perm[off:off + n]
        pt[b, 1, :n] = perm[off:off + n] + numPages
        off += n
        for j in range(L_list[b]):
            kp, vp = pt[b, 0, j // TPP], pt[b, 1, j // TPP]
            pool[kp, j % TPP, :, :D] = k_dense[b, j]
            pool[vp, j % TPP, :, :D] = v_dense[b, j]
            if fill_tails:
                pool[kp, j % TPP, 0, D:] = idxK_dense[b, j]
    return pool, pt


def test_decode_state_equals_prefill_last_row(oracle_mod):
    cfg, t = _small_prefill(B=1, S=260, budget=8)
    _, kbar = _idx(oracle_mod, cfg, t, want_kbar=True)
    for L in (1, 3, 4, 5, 36, 37, 200, 259, 260):
        tt = L - 1
        n_prev = tt // 4
        tail = t["idxK"][0, 4 * n_prev:tt] if tt % 4 else None
        ind, knew, sc = oracle_mod.indexer_decode_state(
            t["idxQ"][0, tt], t["idxK"][0, tt], t["wq"], t["wk"], kbar[0, :n_prev] if n_prev else None, tail,
            L, rot=cfg.rot, ratio=4, budget=cfg.budget, topK=cfg.topK, theta=cfg.theta, eps=cfg.eps)
        ctx = np.array([L], np.int32)
        ref = oracle_mod.indexer_prefill(t["idxQ"], t["idxK"], t["wq"], t["wk"], ctx, rot=cfg.rot, ratio=4,
                                         budget=cfg.budget, topK=cfg.topK, theta=cfg.theta, eps=cfg.eps,
                                         rows=np.array([tt], np.int64))
        assert np.array_equal(ind, ref[0])
        if L % 4 == 0:
            assert np.array_equal(knew.view(np.uint16), kbar[0, L // 4 - 1].view(np.uint16))
        else:
            assert knew is None


def test_decode_pool_passes_match_prefill(oracle_mod):
    Hq, Hkv, D, Hi, di, rot, budget = 4, 2, 128, 4, 64, 32, 8
    topK = budget * 4 + 3
    L_list = [1, 4, 130, 257, 300]
    S = 300
    cfg, t = _small_prefill(B=len(L_list), S=S, Hq=Hq, Hkv=Hkv, D=D, Hi=Hi, di=di, rot=rot, budget=budget)
    ctx = np.array(L_list, np.int32)
    ref_ind, kbar = oracle_mod.indexer_prefill(t["idxQ"], t["idxK"], t["wq"], t["wk"], ctx, rot=rot, ratio=4,
                                               budget=budget, topK=topK, theta=1e4, eps=1e-6, want_kbar=True)
    maxPages = 4
    pool, pt = _pool_from_dense(t["idxK"], t["k"], t["v"], L_list, Hkv, D, di, maxPages, seed=9)
    # the state before decoding token L-1: block keys of blocks complete before it
    for b, L in enumerate(L_list):
        for g in range((L - 1) // 4):
            pool[pt[b, 1, (4 * g) // TPP], (4 * g) % TPP, 0, D:] = kbar[b, g]
    before = pool.copy()
    q_new = np.stack([t["idxQ"][b, L - 1] for b, L in enumerate(L_list)])
    k_new = np.stack([t["idxK"][b, L - 1] for b, L in enumerate(L_list)])
    ind = oracle_mod.indexer_decode(q_new, k_new, t["wq"], t["wk"], pool, pt, ctx, D=D, rot=rot, ratio=4,
                                    budget=budget, topK=topK, theta=1e4, eps=1e-6)
    for b, L in enumerate(L_list):
        assert np.array_equal(ind[b], ref_ind[b, L - 1])
    # exactly one tail changed per sequence
    changed = np.argwhere(~((pool == before) | (np.isnan(pool) & np.isnan(before))))
    for b, L in enumerate(L_list):
        tt = L - 1
        if L % 4 == 0:
            g = L // 4 - 1
            page, slot = pt[b, 1, (4 * g) // TPP], (4 * g) % TPP
            assert np.array_equal(pool[page, slot, 0, D:].view(np.uint16), kbar[b, g].view(np.uint16))
        else:
            page, slot = pt[b, 0, tt // TPP], tt % TPP
            assert np.array_equal(pool[page, slot, 0, D:].view(np.uint16), k_new[b].view(np.uint16))
    assert all(c[2] == 0 and c[3] >= D for c in changed)
    assert len({(c[0], c[1]) for c in changed}) <= len(L_list)
    # attention through the page table equals the dense prefill row
    q_tok = np.stack([t["q"][b, L - 1] for b, L in enumerate(L_list)])
    out = oracle_mod.sparse_decode(q_tok, pool, pt, ind, ctx, D=D, scale=0.088)
    for b, L in enumerate(L_list):
        ref = oracle_mod.sparse_prefill(t["q"], t["k"], t["v"], ref_ind[b:b + 1, L - 1], ctx, 0.088,
                                        rows=np.array([b * S + L - 1], np.int64))
        np.testing.assert_allclose(out[b], ref[0], rtol=0, atol=1e-13)
    # only columns [0, D) of pool rows are read: NaN tails everywhere change nothing
    pool_nan = pool.copy()
    pool_nan[..., D:] = np.nan
    out_nan = oracle_mod.sparse_decode(q_tok, pool_nan, pt, ind, ctx, D=D, scale=0.088)
    np.testing.assert_array_equal(out_nan, out)
    # a different page permutation gives identical outputs
    pool2, pt2 = _pool_from_dense(t["idxK"], t["k"], t["v"], L_list, Hkv, D, di, maxPages, seed=10)
    out2 = oracle_mod.sparse_decode(q_tok, pool2, pt2, ind, ctx, D=D, scale=0.088)
    np.testing.assert_array_equal(out2, out)


# ---------------------------------------------------------------- bf16 inputs
# ("Cute Dsl Qsa Sparse Runner": Q/K/V are fp16 or bf16.)  The bf16 passes
# are pinned to the fp16 ones: on values that both formats hold exactly the
# two must agree to the last bit, and widening must match torch's.

def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)


def _shared_values(shape, rng):
    """Values exact in fp16 and bf16: k/8 with |k| <= 31 (5 significant bits)."""
    return (rng.integers(-31, 32, size=shape) / 8.0).astype(np.float32)


def test_bf16_widening_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_mod.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_attention_equals_fp16_on_shared_values(oracle_mod):
    rng = np.random.default_rng(5)
    B, S, Hq, Hkv, D, topK = 2, 40, 4, 2, 16, 24
    q, k, v = (_shared_values(s, rng) for s in ((B, S, Hq, D), (B, S, Hkv, D), (B, S, Hkv, D)))
    ctx = np.array([40, 29], np.int32)
    ind = np.full((B, S, topK), -1, np.int32)
    for b in range(B):
        for t in range(int(ctx[b])):
            n = min(t + 1, topK)
            ind[b, t, :n] = rng.choice(t + 1, size=n, replace=False)
    o16 = oracle_mod.sparse_prefill(q.astype(np.float16), k.astype(np.float16), v.astype(np.float16), ind, ctx, 0.25)
    ob = oracle_mod.sparse_prefill(_bf16_bits(q), _bf16_bits(k), _bf16_bits(v), ind, ctx, 0.25, bf16=True)
    assert np.array_equal(o16, ob)
    # one index: the (bf16) value row itself
    one = np.full((B, S, topK), -1, np.int32)
    one[:, :, 0] = 3
    v2 = rng.standard_normal((B, S, Hkv, D)).astype(np.float32)
    ob1 = oracle_mod.sparse_prefill(_bf16_bits(q), _bf16_bits(k), _bf16_bits(v2), one, np.array([S, S], np.int32),
                                    0.25, bf16=True)
    vb = torch.from_numpy(v2).to(torch.bfloat16).to(torch.float64).numpy()
    for h in range(Hq):
        assert np.array_equal(ob1[:, 10, h], vb[:, 3, h // (Hq // Hkv)])


def test_bf16_decode_equals_fp16_on_shared_values(oracle_mod):
    rng = np.random.default_rng(6)
    B, Hq, Hkv, D, phd, npg, topK = 2, 8, 2, 16, 24, 6, 40
    pool = _shared_values((npg, 128, Hkv, phd), rng)
    pt = np.stack([np.stack([np.arange(3), np.arange(3) + 3]) for _ in range(B)]).astype(np.int32)
    q = _shared_values((B, Hq, D), rng)
    ctx = np.array([300, 57], np.int32)
    ind = np.full((B, topK), -1, np.int32)
    for b in range(B):
        ind[b, :topK - 5] = rng.choice(int(ctx[b]), size=topK - 5, replace=False)
    o16 = oracle_mod.sparse_decode(q.astype(np.float16), pool.astype(np.float16), pt, ind, ctx, D=D, scale=0.3)
    ob = oracle_mod.sparse_decode(_bf16_bits(q), _bf16_bits(pool), pt, ind, ctx, D=D, scale=0.3, bf16=True)
    assert np.array_equal(o16, ob)


# ------------------------------------------------ upstream q/k norm + RoPE
# ("Qsa Attention Plugin", fused step 1: packed-QKV split, per-head qk-norm
# with (1 + w), partial RoPE.)  Pinned to the index-query prep, which carries
# the RMSNorm and RoPE pins above, and to fp16 round-to-nearest-even.

def test_rope_qkv_heads_positions_and_padding(oracle_mod):
    rng = np.random.default_rng(9)
    B, S, Hq, Hkv, D, rot = 2, 7, 4, 2, 64, 32
    qkv = rng.standard_normal((B, S, Hq + 2 * Hkv, D)).astype(np.float16)
    qw = (0.1 * rng.standard_normal(D)).astype(np.float32)
    kw = (0.1 * rng.standard_normal(D)).astype(np.float32)
    ctx = np.array([7, 4], np.int32)
    q, k, v = oracle_mod.rope_qkv(qkv, qw, kw, ctx, Hq=Hq, Hkv=Hkv, rot=rot, theta=1e4, eps=1e-6)
    for b in range(B):
        for s in range(S):
            if s >= ctx[b]:
                assert not q[b, s].any() and not k[b, s].any() and not v[b, s].any()
                continue
            for h in range(Hq):
                want = oracle_mod.index_q(qkv[b, s, h], qw, rot=rot, pos=s, theta=1e4, eps=1e-6).astype(np.float16)
                assert np.array_equal(q[b, s, h].view(np.uint16), want.view(np.uint16))
            for h in range(Hkv):
                want = oracle_mod.index_q(qkv[b, s, Hq + h], kw, rot=rot, pos=s, theta=1e4, eps=1e-6).astype(np.float16)
                assert np.array_equal(k[b, s, h].view(np.uint16), want.view(np.uint16))
                assert np.array_equal(v[b, s, h].view(np.uint16), qkv[b, s, Hq + Hkv + h].view(np.uint16))
    # one new token (S == 1) sits at position L - 1
    q1, k1, _ = oracle_mod.rope_qkv(qkv[:, :1], qw, kw, np.array([300, 1], np.int32), Hq=Hq, Hkv=Hkv, rot=rot,
                                    theta=1e4, eps=1e-6)
    want = oracle_mod.index_q(qkv[0, 0, 1], qw, rot=rot, pos=299, theta=1e4, eps=1e-6).astype(np.float16)
    assert np.array_equal(q1[0, 0, 1].view(np.uint16), want.view(np.uint16))
    want = oracle_mod.index_q(qkv[1, 0, Hq], kw, rot=rot, pos=0, theta=1e4, eps=1e-6).astype(np.float16)
    assert np.array_equal(k1[1, 0, 0].view(np.uint16), want.view(np.uint16))
