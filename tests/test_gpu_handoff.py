"""Prefill -> decode hand-off of the indexer state through the C ABI.

qsa_indexer_prefill runs on sequences of length L; qsa_indexer_prefill_handoff
writes its block keys and the trailing raw keys into a paged pool
("Qsa Attention Plugin", "KV pool contract"); qsa_indexer_decode then adds the
token at position L.  The pool tails must hold exactly the oracle's block keys
and the raw keys, and the decode list must be the prefill list of row L of the
same sequence extended by that token (oracle), up to ties at the cut."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_qsa_gb300 import _binding as qb
from block_sparse_gqa_qsa_gb300 import synthetic as syn
from qsa_testlib import check_list, compare_selection, f32, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
TPP = syn.TOKENS_PER_PAGE


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_gqa_qsa_gb300 import build
    build.build()
    qb.lib()


CASES = [
    # L = 1 (no complete block), 515 (128 blocks + 3 tail tokens), 2047 (block 511 completes at the new token),
    # 3000 (n_c > budget, and the new token leaves the block incomplete)
    (dataclasses.replace(syn.PREFILL_PARITY, name="handoff", B=4, S=3001, seed=41), (1, 515, 2047, 3000)),
    (dataclasses.replace(syn.PREFILL_PARITY, name="handoff_r8_di64", B=2, S=3001, di=64, rot=32, Hi=4, ratio=8,
                         budget=100, seed=42), (799, 2999)),
]


@pytest.mark.parametrize("cfg,lengths", CASES, ids=[c[0].name for c in CASES])
def test_handoff_then_decode_matches_prefill_row(cfg, lengths):
    L = torch.tensor(lengths, dtype=torch.int32)
    t = syn.make_prefill(cfg, poison=False)  # rows up to L (inclusive) are real data
    t_dev = {k: v.to(DEV) for k, v in t.items()}
    # prefill indexer on the first L tokens of each sequence
    ws = qb.alloc_workspace(qb.indexer_prefill_workspace_size(cfg.B, cfg.S, cfg.di, cfg.ratio), DEV)
    ind = torch.empty((cfg.B, cfg.S, cfg.topK), dtype=torch.int32, device=DEV)
    qb.indexer_prefill(t_dev["idxQ"], t_dev["idxK"], t_dev["wq"], t_dev["wk"], L.to(DEV), ind, ws, rot=cfg.rot,
                       ratio=cfg.ratio, budget=cfg.budget, topK=cfg.topK, theta=cfg.theta, eps=cfg.eps)
    # a paged pool with shuffled pages covering L + 1 tokens
    D, Hkv = 128, 2
    mpp = -(-cfg.S // TPP)
    pages = [-(-(int(x) + 1) // TPP) for x in lengths]
    npg = sum(pages)
    g = torch.Generator().manual_seed(cfg.seed)
    perm = torch.randperm(npg, generator=g).to(torch.int32)
    pt = torch.zeros((cfg.B, 2, mpp), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, 0, :n] = perm[off:off + n]
        pt[b, 1, :n] = perm[off:off + n] + npg
        off += n
    pool = torch.randn((2 * npg, TPP, Hkv, D + cfg.di), generator=g).to(torch.float16).to(DEV)
    pool0 = pool.clone()
    pt_dev = pt.to(DEV)
    qb.indexer_prefill_handoff(t_dev["idxK"], L.to(DEV), ws, pool, pt_dev, D=D, ratio=cfg.ratio)
    torch.cuda.synchronize()
    assert int(to_np(ws[:4]).view(np.int32)[0]) == 0, "workspace status word"

    # the tails: oracle block keys (bit-exact) and raw keys; nothing else changed
    t_np = {k: v.numpy() for k, v in t.items()}
    _, kb_ref = oracle.indexer_prefill(t_np["idxQ"], t_np["idxK"], t_np["wq"], t_np["wk"], L.numpy(), rot=cfg.rot,
                                       ratio=cfg.ratio, budget=cfg.budget, topK=cfg.topK, theta=cfg.theta,
                                       eps=f32(cfg.eps), rows=np.zeros(1, np.int64), want_kbar=True)
    want = pool0.clone()
    for b, Lb in enumerate(lengths):
        n_c = Lb // cfg.ratio
        for gb in range(n_c):
            tok = gb * cfg.ratio
            want[int(pt[b, 1, tok // TPP]), tok % TPP, 0, D:] = torch.from_numpy(kb_ref[b, gb].copy()).to(DEV)
        for tok in range(n_c * cfg.ratio, Lb):
            want[int(pt[b, 0, tok // TPP]), tok % TPP, 0, D:] = t_dev["idxK"][b, tok]
    assert torch.equal(pool.view(torch.int16), want.view(torch.int16))

    # decode the token at position L; its list must be prefill row L of the extended sequence
    pos = L.long()
    bidx = torch.arange(cfg.B)
    idxQ_new = t["idxQ"][bidx, pos].contiguous().to(DEV)
    idxK_new = t["idxK"][bidx, pos].contiguous().to(DEV)
    ctx_new = (L + 1).to(DEV)
    wsd = qb.alloc_workspace(qb.indexer_decode_workspace_size(cfg.B, mpp, cfg.ratio, cfg.budget), DEV)
    dl = torch.full((cfg.B, 1, cfg.topK), 7, dtype=torch.int32, device=DEV)
    qb.indexer_decode(idxQ_new, idxK_new, t_dev["wq"], t_dev["wk"], pool, pt_dev, ctx_new, dl, wsd, D=D, rot=cfg.rot,
                      ratio=cfg.ratio, budget=cfg.budget, topK=cfg.topK, theta=cfg.theta, eps=cfg.eps)
    torch.cuda.synchronize()
    assert int(to_np(wsd[:4]).view(np.int32)[0]) == 0, "decode workspace status word"
    rows = np.array([b * cfg.S + int(x) for b, x in enumerate(lengths)], np.int64)
    ref, sc = oracle.indexer_prefill(t_np["idxQ"], t_np["idxK"], t_np["wq"], t_np["wk"], (L + 1).numpy(), rot=cfg.rot,
                                     ratio=cfg.ratio, budget=cfg.budget, topK=cfg.topK, theta=cfg.theta,
                                     eps=f32(cfg.eps), rows=rows, want_scores=True)
    got = to_np(dl)[:, 0]
    for b, Lb in enumerate(lengths):
        check_list(got[b], Lb, Lb + 1, cfg.ratio, cfg.budget)
        compare_selection(got[b], ref[b], sc[b], Lb, cfg.ratio, cfg.budget)
