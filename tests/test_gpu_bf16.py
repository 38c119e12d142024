"""bf16 surface of the two attention calls ("Cute Dsl Qsa Sparse Runner": the
runners take fp16 or bf16) through the C ABI, against the oracle's bf16 passes.

Tolerance, from the arithmetic of the bf16 path: scores and softmax in fp32
(~1e-6 relative), P rounded to bf16 for the PV product (each weight off by at
most 2^-9 of itself, so o moves by at most 2^-9 * max|v|), output rounded to
bf16 (at most 2^-9 * |o| <= 2^-9 * max|v|):  |o - o_f64| <= 2^-8 * max|v| + 1e-4.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_qsa_gb300 import _binding as qb
from block_sparse_gqa_qsa_gb300 import synthetic as syn
from qsa_testlib import f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_gqa_qsa_gb300 import build
    build.build()
    qb.lib()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _tol(v: torch.Tensor) -> float:
    return 2.0 ** -8 * float(v.float().abs().nan_to_num(0.0).max()) + 1e-4


@pytest.mark.parametrize("impl", ["mma", "tcgen05"])
@pytest.mark.parametrize("Hq,Hkv", [(16, 2), (32, 2)])
def test_sparse_prefill_bf16(Hq, Hkv, impl):
    cfg = dataclasses.replace(syn.PREFILL_PARITY, Hq=Hq, Hkv=Hkv, seed=51 + Hq)
    t = syn.make_prefill(cfg)
    q, k, v = (t[n].float().to(torch.bfloat16) for n in ("q", "k", "v"))  # NaN rows past L stay NaN
    lists = syn.random_lists(cfg.B, cfg.S, cfg.topK, t["ctx"], seed=cfg.seed)
    out = torch.full((cfg.B, cfg.S, cfg.Hq, cfg.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    qb.sparse_prefill(q.to(DEV), k.to(DEV), v.to(DEV), lists.to(DEV), t["ctx"].to(DEV), out, f32(cfg.scale),
                      impl=impl)
    torch.cuda.synchronize()
    ref = oracle.sparse_prefill(_bits(q), _bits(k), _bits(v), lists.numpy(), t["ctx"].numpy(), f32(cfg.scale),
                                bf16=True)
    got = out.float().cpu().numpy()
    ctx = t["ctx"].numpy()
    tol = _tol(v)
    for b in range(cfg.B):
        L = int(ctx[b])
        assert not np.isnan(got[b, :L]).any()
        assert np.abs(got[b, :L] - ref[b, :L]).max() <= tol, (b, np.abs(got[b, :L] - ref[b, :L]).max(), tol)
        assert np.all(_bits(out[b, L:]) == 0), "rows past the live length are exact zeros"
    # a single entry: P = 1 exactly, so o is the bf16 value row bit for bit
    one = torch.full_like(lists, -1)
    one[:, :, 0] = 5
    qb.sparse_prefill(q.to(DEV), k.to(DEV), v.to(DEV), one.to(DEV), t["ctx"].to(DEV), out, f32(cfg.scale),
                      impl=impl)
    torch.cuda.synchronize()
    G = cfg.Hq // cfg.Hkv
    for b in range(cfg.B):
        L = int(ctx[b])
        want = v[b, 5].repeat_interleave(G, dim=0)
        assert torch.equal(out[b, 10:L].cpu().view(torch.int16), want[None].expand(L - 10, -1, -1).view(torch.int16))


def test_sparse_decode_bf16():
    cfg = dataclasses.replace(syn.DECODE_PARITY, Hq=32, Hkv=4, seed=61)
    d = syn.make_decode(cfg)
    pool = d["pool"].float().to(torch.bfloat16)
    q = d["q"].float().to(torch.bfloat16)
    rng = np.random.default_rng(cfg.seed)
    lists = np.full((cfg.B, cfg.topK), -1, np.int32)
    for b, L in enumerate(d["ctx"].numpy()):
        n = min(int(L), cfg.topK - 3)
        lists[b, :n] = rng.choice(int(L), size=n, replace=False)
    po, ps, pc = qb.sparse_decode_workspace_elems(cfg.B, cfg.Hkv, cfg.D)
    ws = (torch.zeros(po, device=DEV), torch.zeros(ps, device=DEV), torch.zeros(pc, dtype=torch.int32, device=DEV))
    out = torch.full((cfg.B, 1, cfg.Hq, cfg.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    qb.sparse_decode(q.to(DEV), pool.to(DEV), d["page_table"].to(DEV), torch.from_numpy(lists[:, None, :]).to(DEV),
                     d["ctx"].to(DEV), out, *ws, D=cfg.D, scale=f32(cfg.scale))
    torch.cuda.synchronize()
    ref = oracle.sparse_decode(_bits(q[:, 0]), _bits(pool), d["page_table"].numpy(), lists, d["ctx"].numpy(), D=cfg.D,
                               scale=f32(cfg.scale), bf16=True)
    got = out[:, 0].float().cpu().numpy()
    assert not np.isnan(got).any()
    assert np.abs(got - ref).max() <= _tol(pool[..., :cfg.D])
    assert int(ws[2].abs().sum()) == 0, "split counters re-armed"
