"""Gather-to-scratch form of the decode through the C ABI (qsa.rs, "qsa_gather"
and the scratch-as-paged-cache note).

qsa_gather_selected copies the K/V rows that a decode list names into
contiguous scratch and describes the scratch as a paged pool (page table,
list, lengths).  The unchanged qsa_sparse_decode on that scratch must return
the same bits as qsa_sparse_decode on the pool with the original list: every
entry keeps its list position, so each split sees the same keys in the same
order.  The result is also held to the oracle's attention bar, and the scratch
rows to the pool rows bit for bit."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_qsa_gb300 import _binding as qb
from block_sparse_gqa_qsa_gb300 import synthetic as syn
from qsa_testlib import check_attention, f32, to_np

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


def _decode(q, pool, pt, lists, ctx, cfg, scale):
    po, ps, pc = qb.sparse_decode_workspace_elems(cfg.B, cfg.Hkv, cfg.D)
    ws = (torch.zeros(po, device=DEV), torch.zeros(ps, device=DEV), torch.zeros(pc, dtype=torch.int32, device=DEV))
    out = torch.full((cfg.B, 1, cfg.Hq, cfg.D), float("nan"), dtype=q.dtype, device=DEV)
    qb.sparse_decode(q, pool, pt, lists, ctx, out, *ws, D=cfg.D, scale=scale)
    return out


def _ab(d_dev, lists_dev, cfg, scale):
    """(in-kernel gathers, gather-to-scratch) outputs and the scratch buffers."""
    a = _decode(d_dev["q"], d_dev["pool"], d_dev["page_table"], lists_dev, d_dev["ctx"], cfg, scale)
    sc = qb.gather_scratch(cfg.B, cfg.Hkv, cfg.D, cfg.topK, dtype=d_dev["pool"].dtype, device=DEV)
    sc[0].fill_(float("nan"))  # unwritten slots must never be read
    qb.gather_selected(d_dev["pool"], d_dev["page_table"], lists_dev, d_dev["ctx"], *sc, D=cfg.D)
    b = _decode(d_dev["q"], sc[0], sc[1], sc[2], sc[3], cfg, scale)
    torch.cuda.synchronize()
    return a, b, sc


def _valid(lists, ctx, pt, nflat):
    """Entries that name a row: inside [0, L) and on K and V pages inside the pool."""
    B, K = lists.shape
    ok = np.zeros((B, K), bool)
    for b in range(B):
        for n, j in enumerate(lists[b]):
            if 0 <= j < ctx[b]:
                kp, vp = pt[b, 0, j // TPP], pt[b, 1, j // TPP]
                ok[b, n] = 0 <= kp < nflat and 0 <= vp < nflat
    return ok


def _check_scratch(sc, d_dev, lists, ctx, cfg):
    scratch, spt, sidx, slen = (to_np(t) if i else t for i, t in enumerate(sc))
    pt = to_np(d_dev["page_table"])
    P = spt.shape[-1]
    ok = _valid(lists, ctx, pt, d_dev["pool"].shape[0])
    assert np.array_equal(sidx[:, 0], np.where(ok, np.arange(cfg.topK)[None, :], -1))
    assert np.all(slen == cfg.topK)
    for b in range(cfg.B):
        assert np.array_equal(spt[b, 0], b * P + np.arange(P)) and np.array_equal(spt[b, 1], (cfg.B + b) * P + np.arange(P))
        n = np.nonzero(ok[b])[0]
        j = torch.from_numpy(lists[b, n].astype(np.int64)).to(DEV)
        pool = d_dev["pool"]
        ptd = d_dev["page_table"]
        want_k = pool[ptd[b, 0, j // TPP].long(), j % TPP, :, :cfg.D]
        want_v = pool[ptd[b, 1, j // TPP].long(), j % TPP, :, :cfg.D]
        nd = torch.from_numpy(n.astype(np.int64)).to(DEV)
        got_k = scratch.view(-1, cfg.Hkv, cfg.D)[b * P * TPP + nd]
        got_v = scratch.view(-1, cfg.Hkv, cfg.D)[(cfg.B + b) * P * TPP + nd]
        assert torch.equal(got_k.view(torch.int16), want_k.view(torch.int16))
        assert torch.equal(got_v.view(torch.int16), want_v.view(torch.int16))


def _to_dev(d):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _np(d):
    return {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


@pytest.mark.parametrize("Hq,Hkv", [(16, 2), (32, 4)])
def test_gather_matches_in_kernel_decode(Hq, Hkv):
    cfg = dataclasses.replace(syn.DECODE_PARITY, Hq=Hq, Hkv=Hkv, seed=71 + Hq)
    d = syn.make_decode(cfg)
    d_np = _np(d)
    lists = oracle.indexer_decode(d_np["idxQ"], d_np["idxK"], d_np["wq"], d_np["wk"], d_np["pool"].copy(),
                                  d_np["page_table"], d_np["ctx"], D=cfg.D, rot=cfg.rot, ratio=cfg.ratio,
                                  budget=cfg.budget, topK=cfg.topK, theta=cfg.theta, eps=f32(cfg.eps))
    d_dev = _to_dev(d)
    lists_dev = torch.from_numpy(lists[:, None, :].copy()).to(DEV)
    a, b, sc = _ab(d_dev, lists_dev, cfg, f32(cfg.scale))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "gather-to-scratch differs from in-kernel gathers"
    ref = oracle.sparse_decode(d_np["q"][:, 0], d_np["pool"], d_np["page_table"], lists, d_np["ctx"], D=cfg.D,
                               scale=f32(cfg.scale))
    check_attention(to_np(b)[:, 0], ref, "gather-to-scratch decode")
    _check_scratch(sc, d_dev, lists, d_np["ctx"], cfg)


def test_gather_holes_invalid_entries_and_bad_pages():
    cfg = dataclasses.replace(syn.DECODE_PARITY, B=4, ctx_list=(0, 700, 1500, 6000), seed=77)
    d = syn.make_decode(cfg)
    rng = np.random.default_rng(3)
    lists = np.full((cfg.B, cfg.topK), -1, np.int32)
    for b, L in enumerate(cfg.ctx_list):
        n = min(L, cfg.topK - 40)
        if n:
            lists[b, :n] = rng.permutation(L)[:n]  # unsorted
    lists[1, 5:25] = -1                            # holes in the middle
    lists[2, 3] = 1500                             # = L: outside the sequence
    lists[2, 7] = -9                               # negative, not -1
    lists[3, 10] = 10 ** 6                         # far outside
    pt = d["page_table"].clone()
    pt[3, 0, 2] = 10 ** 7                          # a K page outside the pool
    d["page_table"] = pt
    d_dev = _to_dev(d)
    lists_dev = torch.from_numpy(lists[:, None, :].copy()).to(DEV)
    a, b, sc = _ab(d_dev, lists_dev, cfg, 0.08)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert np.all(to_np(b)[0].view(np.uint16) == 0), "L = 0: zero output"
    _check_scratch(sc, d_dev, lists, d["ctx"].numpy(), cfg)
    # the oracle on the sequences whose pages are all inside the pool; entries outside [0, L) are skipped
    # (read as -1), which is how the kernels treat them
    d_np = _np(d)
    live = np.where((lists >= 0) & (lists < d_np["ctx"][:, None]), lists, -1).astype(np.int32)
    ref = oracle.sparse_decode(d_np["q"][:3, 0], d_np["pool"], d_np["page_table"][:3], live[:3], d_np["ctx"][:3],
                               D=cfg.D, scale=f32(0.08))
    check_attention(to_np(b)[:3, 0], ref, "holes and invalid entries")


def test_gather_bf16_pool():
    cfg = dataclasses.replace(syn.DECODE_PARITY, Hq=32, Hkv=4, seed=79)
    d = syn.make_decode(cfg)
    rng = np.random.default_rng(4)
    lists = np.full((cfg.B, cfg.topK), -1, np.int32)
    for b, L in enumerate(d["ctx"].numpy()):
        n = min(int(L), cfg.topK - 3)
        lists[b, :n] = np.sort(rng.choice(int(L), size=n, replace=False))
    d_dev = _to_dev(d)
    d_dev["pool"] = d_dev["pool"].to(torch.bfloat16)
    d_dev["q"] = d_dev["q"].to(torch.bfloat16)
    lists_dev = torch.from_numpy(lists[:, None, :].copy()).to(DEV)
    a, b, sc = _ab(d_dev, lists_dev, cfg, f32(cfg.scale))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    _check_scratch(sc, d_dev, lists, d["ctx"].numpy(), cfg)


def test_gather_full_size_decode_32():
    cfg = syn.DECODE_32
    d = syn.make_decode(cfg, device=DEV)
    d_dev = _to_dev(d)
    ctx = d["ctx"].cpu().numpy()
    rng = np.random.default_rng(5)
    lists = np.full((cfg.B, cfg.topK), -1, np.int32)
    for b, L in enumerate(ctx):  # ascending lists of the method's full width
        n = min(int(L), cfg.topK)
        lists[b, :n] = np.sort(rng.choice(int(L), size=n, replace=False))
    lists_dev = torch.from_numpy(lists[:, None, :].copy()).to(DEV)
    a, b, sc = _ab(d_dev, lists_dev, cfg, f32(cfg.scale))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    spt, sidx = to_np(sc[1]), to_np(sc[2])[:, 0]
    assert np.array_equal(sidx, np.where(lists >= 0, np.arange(cfg.topK)[None, :], -1))
    q = to_np(d_dev["q"])
    for bb in (0, cfg.B - 1):  # sampled sequences against the oracle, rows taken from the scratch
        n = np.nonzero(lists[bb] >= 0)[0]
        P = spt.shape[-1]
        rows = sc[0].view(-1, cfg.Hkv, cfg.D)
        kr = to_np(rows[bb * P * TPP + torch.from_numpy(n).to(DEV)])
        vr = to_np(rows[(cfg.B + bb) * P * TPP + torch.from_numpy(n).to(DEV)])
        ref = oracle.attend_rows(q[bb, 0], kr, vr, f32(cfg.scale))
        check_attention(to_np(b)[bb, 0], ref, f"{cfg.name} seq {bb}")
