"""The upstream q/k norm + partial RoPE of packed QKV (qsa_rope_qkv) through the
C ABI against the oracle ("Qsa Attention Plugin", fused step 1).

The GPU evaluates the norm and the rotation in fp32 and rounds once to fp16;
the oracle rounds the f64 value once.  The fp32 evaluation is off by a few
units of 2^-24 of its operands (normalised values, |y| <= ~5), about 1e-6
absolute, so the two fp16 results differ by at most one fp16 ulp plus that
error (which exceeds an ulp only where the rotation nearly cancels): the bar
is |got - want| <= ulp(want) + 2^-18, with exact equality for almost all
values.  V heads, padding rows, pool placement and the pool tails are
bit-exact."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_qsa_gb300 import _binding as qb
from block_sparse_gqa_qsa_gb300 import synthetic as syn

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


def _close_fp16(got: np.ndarray, want: np.ndarray):
    g, w = got.astype(np.float64), want.astype(np.float64)
    bar = np.spacing(np.abs(want)).astype(np.float64) + 2.0 ** -18
    assert np.all(np.abs(g - w) <= bar), float(np.max(np.abs(g - w) - bar))
    assert np.mean(got.view(np.uint16) == want.view(np.uint16)) > 0.99


# rot = 0 .. D covers every partner distance (0, 1, 2, 4, 8 chunks); Hq 64 + 2 * 8 heads at D 128 is 1280
# chunks per token, more than one load batch of the CTA
@pytest.mark.parametrize("D,rot,Hq,Hkv", [(128, 64, 8, 2), (64, 32, 8, 2), (128, 128, 4, 1), (128, 16, 8, 2),
                                          (64, 0, 4, 2), (128, 64, 64, 8)])
def test_rope_qkv_prefill_dense(D, rot, Hq, Hkv):
    B, S = 2, 2000  # 4000 tokens: several per CTA of the persistent grid, so the copy ring wraps
    g = torch.Generator().manual_seed(71 + D)
    qkv = torch.randn((B, S, Hq + 2 * Hkv, D), generator=g).to(torch.float16)
    wq = (0.1 * torch.randn(D, generator=g)).float()
    wk = (0.1 * torch.randn(D, generator=g)).float()
    ctx = torch.tensor([2000, 1173], dtype=torch.int32)
    q = torch.full((B, S, Hq, D), float("nan"), dtype=torch.float16, device=DEV)
    k = torch.full((B, S, Hkv, D), float("nan"), dtype=torch.float16, device=DEV)
    v = torch.full((B, S, Hkv, D), float("nan"), dtype=torch.float16, device=DEV)
    qb.rope_qkv(qkv.to(DEV), wq.to(DEV), wk.to(DEV), ctx.to(DEV), q, Hq=Hq, Hkv=Hkv, rot=rot, theta=1e4, eps=1e-6,
                k_out=k, v_out=v)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.rope_qkv(qkv.numpy(), wq.numpy(), wk.numpy(), ctx.numpy(), Hq=Hq, Hkv=Hkv, rot=rot,
                                 theta=1e4, eps=np.float64(np.float32(1e-6)))
    gq, gk, gv = (t.cpu().numpy() for t in (q, k, v))
    _close_fp16(gq, rq)
    _close_fp16(gk, rk)
    assert np.array_equal(gv.view(np.uint16), rv.view(np.uint16))
    assert not gq[1, 1173:].view(np.uint16).any() and not gk[1, 1173:].view(np.uint16).any()
    assert not gv[1, 1173:].view(np.uint16).any()


def test_rope_qkv_decode_into_pool():
    B, Hq, Hkv, D, di, rot = 3, 8, 2, 128, 128, 64
    lengths = (1, 200, 5000)  # the new token at positions 0, 199, 4999
    g = torch.Generator().manual_seed(81)
    qkv = torch.randn((B, 1, Hq + 2 * Hkv, D), generator=g).to(torch.float16)
    wq = (0.1 * torch.randn(D, generator=g)).float()
    wk = (0.1 * torch.randn(D, generator=g)).float()
    ctx = torch.tensor(lengths, dtype=torch.int32)
    pages = [-(-L // TPP) for L in lengths]
    npg, mpp = sum(pages), max(pages)
    perm = torch.randperm(npg, generator=g).to(torch.int32)
    pt = torch.zeros((B, 2, mpp), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, 0, :n] = perm[off:off + n]
        pt[b, 1, :n] = perm[off:off + n] + npg
        off += n
    pool = torch.randn((2 * npg, TPP, Hkv, D + di), generator=g).to(torch.float16).to(DEV)
    pool0 = pool.clone()
    q = torch.empty((B, 1, Hq, D), dtype=torch.float16, device=DEV)
    k = torch.empty((B, 1, Hkv, D), dtype=torch.float16, device=DEV)
    qb.rope_qkv(qkv.to(DEV), wq.to(DEV), wk.to(DEV), ctx.to(DEV), q, Hq=Hq, Hkv=Hkv, rot=rot, theta=1e4,
                eps=1e-6, k_out=k, pool=pool, page_table=pt.to(DEV))
    torch.cuda.synchronize()
    rq, rk, rv = oracle.rope_qkv(qkv.numpy(), wq.numpy(), wk.numpy(), ctx.numpy(), Hq=Hq, Hkv=Hkv, rot=rot,
                                 theta=1e4, eps=np.float64(np.float32(1e-6)))
    _close_fp16(q.cpu().numpy(), rq)
    _close_fp16(k.cpu().numpy(), rk)
    want = pool0.clone()
    for b, L in enumerate(lengths):
        pos = L - 1
        want[int(pt[b, 0, pos // TPP]), pos % TPP, :, :D] = k[b, 0]  # the K rows hold what kOut holds
        want[int(pt[b, 1, pos // TPP]), pos % TPP, :, :D] = torch.from_numpy(rv[b, 0].copy()).to(DEV)
    assert torch.equal(pool.view(torch.int16), want.view(torch.int16)), "only the new tokens' leading columns change"
