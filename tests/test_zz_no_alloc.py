"""qsa_sparse_decode_noalloc: split-K sparse decode on the library's own fixed
scratch, called through the C ABI, against qsa_sparse_decode with a caller
workspace on the same inputs (and the fp64 oracle on the small shape).  The
file sorts last so that the entry point also runs after every other test has
used the library in this process; it passes alone as well."""
from __future__ import annotations

import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_qsa_gb300 import _binding as qb
from block_sparse_gqa_qsa_gb300 import synthetic as syn
from qsa_testlib import check_attention, f32, to_np

DEV = "cuda"


@pytest.fixture(scope="module")
def binding():
    from block_sparse_gqa_qsa_gb300 import build
    build.build()
    qb.lib()
    return qb


def test_noalloc_rejects_before_launch(binding):
    """Host-side checks only: nothing here reaches the GPU."""
    L = binding.lib()
    fake = 1 << 20  # never dereferenced
    p = binding.QsaSparseDecodeParams(qPtr=fake, kvPoolPtr=fake, pageTable=fake, indices=fake, contextLengths=fake,
                                      oPtr=fake, partialO=fake, partialStats=None, splitCounters=None, batchSize=8,
                                      numQHeads=64, numKVHeads=8, headDim=128, poolHeadDim=256, numFlatPages=10,
                                      maxPagesPerSeq=16, topK=2051, attentionScale=0.1)
    assert L.qsa_sparse_decode_noalloc(None) == binding.QSA_ERR_INVALID_ARG
    assert L.qsa_sparse_decode_noalloc(ctypes.byref(p)) == binding.QSA_ERR_INVALID_ARG
    assert b"must be NULL" in L.qsa_last_error_message()
    p.partialO = None
    p.batchSize, p.numKVHeads, p.numQHeads = 257, 1, 8
    assert L.qsa_sparse_decode_noalloc(ctypes.byref(p)) == binding.QSA_ERR_UNSUPPORTED
    msg = L.qsa_last_error_message()
    assert b"257" in msg and b"256" in msg


def _lists(ctx, topK, seed):
    """Distinct live token ids per sequence in random order, -1 padded."""
    rng = np.random.default_rng(seed)
    out = np.full((len(ctx), 1, topK), -1, np.int32)
    for b, L in enumerate(ctx):
        n = min(int(L), topK - 3)
        if n > 0:
            out[b, 0, :n] = rng.choice(int(L), size=n, replace=False)
    return out


def _with_workspace(d_dev, lists_dev, cfg):
    po, ps, pc = qb.sparse_decode_workspace_elems(cfg.B, cfg.Hkv, cfg.D)
    ws = (torch.zeros(po, dtype=torch.float32, device=DEV), torch.zeros(ps, dtype=torch.float32, device=DEV),
          torch.zeros(pc, dtype=torch.int32, device=DEV))
    out = torch.full((cfg.B, 1, cfg.Hq, cfg.D), float("nan"), dtype=torch.float16, device=DEV)
    qb.sparse_decode(d_dev["q"], d_dev["pool"], d_dev["page_table"], lists_dev, d_dev["ctx"], out, *ws, D=cfg.D,
                     scale=f32(cfg.scale))
    return out


def _noalloc(d_dev, lists_dev, cfg):
    out = torch.full((cfg.B, 1, cfg.Hq, cfg.D), float("nan"), dtype=torch.float16, device=DEV)
    qb.sparse_decode_noalloc(d_dev["q"], d_dev["pool"], d_dev["page_table"], lists_dev, d_dev["ctx"], out, D=cfg.D,
                             scale=f32(cfg.scale))
    return out


CASES = [
    # several splits, ragged lengths, an almost empty sequence
    syn.DECODE_PARITY,
    # exactly the scratch capacity: 32 sequences x 8 KV heads = 256 pairs
    dataclasses.replace(syn.DECODE_PARITY, name="noalloc_capacity", B=32, Hq=64, Hkv=8, ctx_list=None,
                        ctx_lo=1, ctx_hi=3000, max_ctx=3072, seed=23),
]


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_noalloc_matches_workspace_entry_twice(binding, cfg):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = syn.make_decode(cfg)
    d_dev = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    lists = _lists(d["ctx"].numpy(), cfg.topK, cfg.seed)
    lists_dev = torch.from_numpy(lists).to(DEV)
    ref = _with_workspace(d_dev, lists_dev, cfg)
    for call in range(2):  # the second call runs on the counters the first one re-armed
        out = _noalloc(d_dev, lists_dev, cfg)
        torch.cuda.synchronize()
        assert not torch.isnan(out).any(), f"call {call}: output not written"
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call}: differs from the workspace entry"
    if cfg.B <= 8:
        d_np = {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        want = oracle.sparse_decode(d_np["q"][:, 0], d_np["pool"], d_np["page_table"], lists[:, 0], d_np["ctx"],
                                    D=cfg.D, scale=f32(cfg.scale))
        check_attention(to_np(out)[:, 0], want, "noalloc decode")


@pytest.mark.gpu
def test_noalloc_small_after_capacity(binding):
    """The shared scratch after a call at full capacity (256 (sequence, KV
    head) pairs, the most its partial slots hold): a smaller call with other
    shapes, and so another slice count, must find its counters at zero and
    match the workspace entry."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    runs = []
    for cfg in (CASES[1], CASES[0]):
        d = syn.make_decode(cfg)
        d_dev = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        lists_dev = torch.from_numpy(_lists(d["ctx"].numpy(), cfg.topK, cfg.seed)).to(DEV)
        runs.append((cfg, d_dev, lists_dev, _noalloc(d_dev, lists_dev, cfg)))
    torch.cuda.synchronize()
    for cfg, d_dev, lists_dev, out in runs:
        ref = _with_workspace(d_dev, lists_dev, cfg)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"{cfg.name}: differs from the workspace entry"
