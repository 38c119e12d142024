"""GPU parity of the decode path through the C ABI: qsa_indexer_decode (state
update in the pool tails, then scoring, selection and expansion) and the
split-K qsa_sparse_decode, against the fp64 CPU oracle."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_qsa_gb300 import _binding as qb
from block_sparse_gqa_qsa_gb300 import synthetic as syn
from qsa_testlib import check_attention, check_list, compare_selection, f32, to_np

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


def _gpu_indexer(d_dev, cfg, ws=None):
    B = cfg.B
    if ws is None:
        ws = qb.alloc_workspace(qb.indexer_decode_workspace_size(B, cfg.maxPagesPerSeq, cfg.ratio, cfg.budget), DEV)
    ind = torch.full((B, 1, cfg.topK), 7, dtype=torch.int32, device=DEV)
    qb.indexer_decode(d_dev["idxQ"], d_dev["idxK"], d_dev["wq"], d_dev["wk"], d_dev["pool"], d_dev["page_table"],
                      d_dev["ctx"], ind, ws, D=cfg.D, rot=cfg.rot, ratio=cfg.ratio, budget=cfg.budget, topK=cfg.topK,
                      theta=cfg.theta, eps=cfg.eps)
    torch.cuda.synchronize()
    return ind, ws


def _gpu_attention(d_dev, lists_dev, cfg, scale, ws=None):
    B = cfg.B
    if ws is None:
        po, ps, pc = qb.sparse_decode_workspace_elems(B, cfg.Hkv, cfg.D)
        ws = (torch.zeros(po, dtype=torch.float32, device=DEV), torch.zeros(ps, dtype=torch.float32, device=DEV),
              torch.zeros(pc, dtype=torch.int32, device=DEV))
    out = torch.full((B, 1, cfg.Hq, cfg.D), float("nan"), dtype=torch.float16, device=DEV)
    qb.sparse_decode(d_dev["q"], d_dev["pool"], d_dev["page_table"], lists_dev, d_dev["ctx"], out, *ws, D=cfg.D,
                     scale=scale)
    torch.cuda.synchronize()
    return out, ws


def _to_dev(d):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _oracle_indexer(d_np, pool_np, cfg):
    ind, sc = oracle.indexer_decode(d_np["idxQ"], d_np["idxK"], d_np["wq"], d_np["wk"], pool_np, d_np["page_table"],
                                    d_np["ctx"], D=cfg.D, rot=cfg.rot, ratio=cfg.ratio, budget=cfg.budget,
                                    topK=cfg.topK, theta=cfg.theta, eps=f32(cfg.eps), want_scores=True)
    return ind, sc


def _np(d):
    return {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


DECODE_SHAPES = [
    syn.DECODE_PARITY,
    # 16 and 8 block keys per page (a short swizzled tile), blocks completed at L % r == 0
    dataclasses.replace(syn.DECODE_PARITY, name="ratio8", ratio=8, ctx_list=(1, 8, 1031, 2048, 4103, 6000), seed=31),
    dataclasses.replace(syn.DECODE_PARITY, name="ratio16", ratio=16, ctx_list=(1, 16, 2063, 4096, 4111, 6000),
                        seed=32),
    # 64-dim index keys (one 64-dim TMA box per page row), fewer index heads
    dataclasses.replace(syn.DECODE_PARITY, name="di64", di=64, rot=32, Hi=4, seed=33),
]


@pytest.mark.parametrize("cfg", DECODE_SHAPES, ids=lambda c: c.name)
def test_indexer_decode_parity_and_state_update(cfg):
    d = syn.make_decode(cfg)
    d_np = _np(d)
    pool_np = d_np["pool"].copy()
    d_dev = _to_dev(d)
    ind, ws = _gpu_indexer(d_dev, cfg)
    ref, sc = _oracle_indexer(d_np, pool_np, cfg)
    g = to_np(ind)[:, 0]
    for b in range(cfg.B):
        L = int(d_np["ctx"][b])
        check_list(g[b], L - 1, L, cfg.ratio, cfg.budget)
        compare_selection(g[b], ref[b], sc[b], L - 1, cfg.ratio, cfg.budget)
    # the pool after the step: identical bytes (tails of head 0 only were written)
    assert np.array_equal(to_np(d_dev["pool"]).view(np.uint16), pool_np.view(np.uint16))
    assert not np.array_equal(pool_np.view(np.uint16), d_np["pool"].view(np.uint16))
    assert int(to_np(ws[:4]).view(np.int32)[0]) == 0, "workspace status word"
    assert qb.last_device_error(ws) == 0, "status word through qsa_last_device_error"
    # a second call on the updated state gives the same lists and leaves the pool unchanged
    ind2, _ = _gpu_indexer(d_dev, cfg, ws)
    assert torch.equal(ind2, ind)
    assert np.array_equal(to_np(d_dev["pool"]).view(np.uint16), pool_np.view(np.uint16))


def test_indexer_decode_edges():
    """Dense rows (n_c <= budget), L = 0, a block completed on a page boundary, ties."""
    cfg = dataclasses.replace(syn.DECODE_PARITY, B=5, budget=40, ctx_list=(0, 3, 128, 160, 4096), max_ctx=4096,
                              seed=21)
    d = syn.make_decode(cfg)
    d_np = _np(d)
    pool_np = d_np["pool"].copy()
    d_dev = _to_dev(d)
    ind, _ = _gpu_indexer(d_dev, cfg)
    ref, sc = _oracle_indexer(d_np, pool_np, cfg)
    g = to_np(ind)[:, 0]
    assert np.all(g[0] == -1)
    for b in range(1, cfg.B):
        L = int(d_np["ctx"][b])
        check_list(g[b], L - 1, L, cfg.ratio, cfg.budget)
        compare_selection(g[b], ref[b], sc[b], L - 1, cfg.ratio, cfg.budget)
    assert np.array_equal(to_np(d_dev["pool"]).view(np.uint16), pool_np.view(np.uint16))
    # exact ties: every block-key tail identical and no RoPE -> lowest ids on both sides
    cfg0 = dataclasses.replace(cfg, rot=0, ctx_list=(3001, 4000, 2, 515, 4095))
    d = syn.make_decode(cfg0)
    pool = d["pool"]
    pool[:, :, 0, cfg0.D:] = pool[0, 0, 0, cfg0.D:]
    d_np = _np(d)
    pool_np = d_np["pool"].copy()
    d_dev = _to_dev(d)
    ind, _ = _gpu_indexer(d_dev, cfg0)
    ref, _ = _oracle_indexer(d_np, pool_np, cfg0)
    assert np.array_equal(to_np(ind)[:, 0], ref)
    # the same ties over more candidates than the selection stages on chip (n_c = 6000 and 5120 blocks,
    # several slices): the final pass reads them back from the workspace
    cfg1 = dataclasses.replace(cfg0, B=2, ctx_list=(24000, 20483), max_ctx=24576, seed=22)
    d = syn.make_decode(cfg1)
    pool = d["pool"]
    pool[:, :, 0, cfg1.D:] = pool[0, 0, 0, cfg1.D:]
    d_np = _np(d)
    pool_np = d_np["pool"].copy()
    d_dev = _to_dev(d)
    ind, _ = _gpu_indexer(d_dev, cfg1)
    ref, _ = _oracle_indexer(d_np, pool_np, cfg1)
    assert np.array_equal(to_np(ind)[:, 0], ref)
    # ties over more than 8 slices of 2048 blocks (n_c = 17500 and 16501): one CTA per slice, and the
    # last one reads the 17500 candidates back from the workspace
    cfg2 = dataclasses.replace(cfg0, B=2, ctx_list=(70000, 66007), max_ctx=70016, seed=24)
    d = syn.make_decode(cfg2)
    pool = d["pool"]
    pool[:, :, 0, cfg2.D:] = pool[0, 0, 0, cfg2.D:]
    d_np = _np(d)
    pool_np = d_np["pool"].copy()
    d_dev = _to_dev(d)
    ind, _ = _gpu_indexer(d_dev, cfg2)
    ref, _ = _oracle_indexer(d_np, pool_np, cfg2)
    assert np.array_equal(to_np(ind)[:, 0], ref)


def test_indexer_decode_bad_page_sets_status_bit():
    """A V page id outside the pool: the scorer's range check skips it and sets bit 1 of the status word,
    read back through qsa_last_device_error; the call itself still returns QSA_OK."""
    cfg = syn.DECODE_PARITY
    d = syn.make_decode(cfg)
    num_pages = d["pool"].shape[0]
    d["page_table"][5, 1, 0] = num_pages + 7  # sequence 5 (L = 6000): its first page holds block keys
    d_dev = _to_dev(d)
    _, ws = _gpu_indexer(d_dev, cfg)
    assert qb.last_device_error(ws) & 2, "bit 1 (page id outside the pool) must be set"
    assert not qb.last_device_error(ws) & 1, "no wait may time out"


def test_indexer_decode_wait_timeout_sets_status_bit():
    """The device-side error path of the page stream: with its progress waits bounded to 1 ns they run
    out, the scorer stops early and records bit 0 of the status word instead of hanging; the call itself
    returns QSA_OK.  Copies already in flight are still waited for (their own 0.2 s bound), so the
    context stays usable: with the default bound restored and a zero-filled workspace, the next call
    matches the oracle with a clean status word."""
    # 4 sequences of 256K tokens: 8192 pages of block keys, ~54 per scorer CTA, more than its 22-stage
    # ring, so right after filling the ring the producer waits on a page its consumers cannot have
    # released yet, and gives up
    cfg = dataclasses.replace(syn.DECODE_PARITY, B=4, Hkv=1, Hq=8, ctx_list=(262144,) * 4, max_ctx=262144, seed=41)
    d = syn.make_decode(cfg, device=DEV)
    d_dev = _to_dev(d)
    try:
        qb.debug_set_wait_limit_ns(1)
        _, ws = _gpu_indexer(d_dev, cfg)
    finally:
        qb.debug_set_wait_limit_ns(0)
    assert qb.last_device_error(ws) & 1, "bit 0 (a wait ran out) must be set"
    torch.cuda.synchronize()  # the context is still usable
    cfg2 = syn.DECODE_PARITY
    d2 = syn.make_decode(cfg2)
    d2_np = _np(d2)
    pool_np = d2_np["pool"].copy()
    d2_dev = _to_dev(d2)
    ind, ws2 = _gpu_indexer(d2_dev, cfg2)
    ref, sc = _oracle_indexer(d2_np, pool_np, cfg2)
    g = to_np(ind)[:, 0]
    for b in range(cfg2.B):
        L = int(d2_np["ctx"][b])
        compare_selection(g[b], ref[b], sc[b], L - 1, cfg2.ratio, cfg2.budget)
    assert qb.last_device_error(ws2) == 0


def _state(pool, pt, b, L, cfg):
    """Compact indexer state of sequence b before decoding token L-1 (torch gathers of input data)."""
    t = L - 1
    n_prev = t // cfg.ratio
    tok = torch.arange(n_prev, device=pool.device) * cfg.ratio
    kb = pool[pt[b, 1, tok // TPP].long(), tok % TPP, 0, cfg.D:cfg.D + cfg.di]
    first = n_prev * cfg.ratio
    tt = torch.arange(first, t, device=pool.device)
    tail = pool[pt[b, 0, tt // TPP].long(), tt % TPP, 0, cfg.D:cfg.D + cfg.di]
    return to_np(kb), to_np(tail)


def _rows(pool, pt, b, lst, cfg):
    j = torch.from_numpy(lst[lst >= 0].astype(np.int64)).to(pool.device)
    kr = pool[pt[b, 0, j // TPP].long(), j % TPP, :, :cfg.D]
    vr = pool[pt[b, 1, j // TPP].long(), j % TPP, :, :cfg.D]
    return to_np(kr), to_np(vr)


# The largest decode batch (1024): every 16th sequence holds ~2000 tokens and the others 1-3, which have
# no complete block.  A scorer CTA's pages then span up to 17 sequences, so the queries of those past its
# shared-memory cache of 8 are read from the workspace.
DECODE_SPARSE = dataclasses.replace(
    syn.DECODE_PARITY, name="decode_B1024_sparse_pages", B=1024, max_ctx=2048, seed=71,
    ctx_list=tuple(2000 + b % 5 if b % 16 == 0 else 1 + b % 3 for b in range(1024)))


@pytest.mark.parametrize("cfg", [syn.DECODE_32, syn.DECODE_LONG, DECODE_SPARSE], ids=lambda c: c.name)
def test_decode_full_size(cfg):
    d = syn.make_decode(cfg, device=DEV)
    d_dev = _to_dev(d)
    pool, pt = d_dev["pool"], d_dev["page_table"]
    ctx = d["ctx"].numpy()
    d_np = _np({k: v for k, v in d.items() if k != "pool"})
    # oracle on the compact state of every sequence, taken before the GPU updates the tails
    ref_lists, ref_new, ref_sc = [], [], []
    for b in range(cfg.B):
        kb, tail = _state(pool, pt, b, int(ctx[b]), cfg)
        lst, knew, sc = oracle.indexer_decode_state(d_np["idxQ"][b], d_np["idxK"][b], d_np["wq"], d_np["wk"], kb,
                                                    tail if len(tail) else None, int(ctx[b]), rot=cfg.rot,
                                                    ratio=cfg.ratio, budget=cfg.budget, topK=cfg.topK,
                                                    theta=cfg.theta, eps=f32(cfg.eps))
        ref_lists.append(lst)
        ref_new.append(knew)
        ref_sc.append(sc)
    ind, ws = _gpu_indexer(d_dev, cfg)
    g = to_np(ind)[:, 0]
    for b in range(cfg.B):
        L = int(ctx[b])
        check_list(g[b], L - 1, L, cfg.ratio, cfg.budget)
        compare_selection(g[b], ref_lists[b], ref_sc[b], L - 1, cfg.ratio, cfg.budget)
        t = L - 1
        if ref_new[b] is not None:  # completed block: its key in the V-row tail of its first token
            first = (L // cfg.ratio - 1) * cfg.ratio
            got = pool[pt[b, 1, first // TPP].long(), first % TPP, 0, cfg.D:cfg.D + cfg.di]
            assert np.array_equal(to_np(got).view(np.uint16), ref_new[b].view(np.uint16))
        else:  # raw key in token t's K-row tail
            got = pool[pt[b, 0, t // TPP].long(), t % TPP, 0, cfg.D:cfg.D + cfg.di]
            assert np.array_equal(to_np(got).view(np.uint16), d_np["idxK"][b].view(np.uint16))
    assert int(to_np(ws[:4]).view(np.int32)[0]) == 0
    # attention over the oracle's lists
    lists_dev = torch.from_numpy(np.stack(ref_lists)[:, None, :]).to(DEV)
    out, _ = _gpu_attention(d_dev, lists_dev, cfg, f32(cfg.scale))
    for b in range(cfg.B):
        kr, vr = _rows(pool, pt, b, ref_lists[b], cfg)
        ref = oracle.attend_rows(d_np["q"][b, 0], kr, vr, f32(cfg.scale))
        check_attention(to_np(out)[b, 0], ref, f"{cfg.name} seq {b}")


@pytest.mark.parametrize("Hq,Hkv", [(16, 2), (32, 4), (32, 2), (12, 1)])
def test_sparse_decode_parity(Hq, Hkv):
    cfg = dataclasses.replace(syn.DECODE_PARITY, Hq=Hq, Hkv=Hkv, seed=Hq + Hkv)
    d = syn.make_decode(cfg)
    d_np = _np(d)
    lists = oracle.indexer_decode(d_np["idxQ"], d_np["idxK"], d_np["wq"], d_np["wk"], d_np["pool"].copy(),
                                  d_np["page_table"], d_np["ctx"], D=cfg.D, rot=cfg.rot, ratio=cfg.ratio,
                                  budget=cfg.budget, topK=cfg.topK, theta=cfg.theta, eps=f32(cfg.eps))
    d_dev = _to_dev(d)
    lists_dev = torch.from_numpy(lists[:, None, :].copy()).to(DEV)
    out, ws = _gpu_attention(d_dev, lists_dev, cfg, f32(cfg.scale))
    ref = oracle.sparse_decode(d_np["q"][:, 0], d_np["pool"], d_np["page_table"], lists, d_np["ctx"], D=cfg.D,
                               scale=f32(cfg.scale))
    check_attention(to_np(out)[:, 0], ref, "decode parity")
    assert int(ws[2].abs().sum()) == 0, "split counters must be re-armed to zero"
    out2, _ = _gpu_attention(d_dev, lists_dev, cfg, f32(cfg.scale), ws)
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16)), "back-to-back calls must agree bitwise"
    # only columns [0, D) are read: NaN tails change nothing
    d_dev["pool"][..., cfg.D:] = float("nan")
    out3, _ = _gpu_attention(d_dev, lists_dev, cfg, f32(cfg.scale), ws)
    assert torch.equal(out3.view(torch.int16), out.view(torch.int16))


@pytest.mark.parametrize("B", [40, 80, 96, 300])
def test_sparse_decode_slice_count_follows_the_batch(B):
    """The slices per (sequence, KV head) follow the batch: at most 8, as many
    as fit one wave of resident CTAs, then the fewest with the same longest
    slice.  With a 4-tile list these batches take 4, 2, 1 and (past one wave
    at any count) 4 slices on a 152-SM GPU.  Each matches the oracle, leaves
    its counters at zero and repeats bit for bit."""
    cfg = dataclasses.replace(syn.DECODE_PARITY, name=f"slices_B{B}", B=B, Hq=32, Hkv=4, Hi=4, di=64, rot=32,
                              budget=63, ctx_lo=1, ctx_hi=300, max_ctx=384, ctx_list=None, seed=60 + B)
    assert cfg.topK == 255
    d = syn.make_decode(cfg, device=DEV)
    d_dev = _to_dev(d)
    pool, pt = d_dev["pool"], d_dev["page_table"]
    ctx = d["ctx"].numpy()
    rng = np.random.default_rng(B)
    lists = np.full((B, cfg.topK), -1, np.int32)
    for b in range(B):
        L = int(ctx[b])
        lists[b, :min(L, cfg.topK)] = np.sort(rng.permutation(L)[:cfg.topK])
    lists_dev = torch.from_numpy(lists[:, None, :].copy()).to(DEV)
    out, ws = _gpu_attention(d_dev, lists_dev, cfg, f32(cfg.scale))
    o, q = to_np(out)[:, 0], to_np(d_dev["q"])[:, 0]
    for b in range(B):
        kr, vr = _rows(pool, pt, b, lists[b], cfg)
        check_attention(o[b], oracle.attend_rows(q[b], kr, vr, f32(cfg.scale)), f"B={B} seq {b}")
    assert int(ws[2].abs().sum()) == 0, "split counters must be re-armed to zero"
    out2, _ = _gpu_attention(d_dev, lists_dev, cfg, f32(cfg.scale), ws)
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16)), "back-to-back calls must agree bitwise"


def test_sparse_decode_page_permutation_and_empty():
    cfg = dataclasses.replace(syn.DECODE_PARITY, B=3, ctx_list=(0, 700, 1500), max_ctx=1536, seed=5)
    d = syn.make_decode(cfg)
    d_np = _np(d)
    rng = np.random.default_rng(1)
    lists = np.full((cfg.B, cfg.topK), -1, np.int32)
    for b, L in enumerate(cfg.ctx_list):
        n = min(L, 450)
        lists[b, :n] = rng.permutation(L)[:n]
    d_dev = _to_dev(d)
    lists_dev = torch.from_numpy(lists[:, None, :].copy()).to(DEV)
    out, ws = _gpu_attention(d_dev, lists_dev, cfg, 0.08)
    o = to_np(out)[:, 0]
    assert np.all(o[0].view(np.uint16) == 0), "L = 0: zero output"
    ref = oracle.sparse_decode(d_np["q"][:, 0], d_np["pool"], d_np["page_table"], lists, d_np["ctx"], D=cfg.D,
                               scale=f32(0.08))
    check_attention(o, ref, "random lists")
    # the same logical cache under another page permutation
    npg = d["num_pages"]
    perm = torch.from_numpy(rng.permutation(npg)).to(DEV)
    mapping = torch.cat([perm, perm + npg])  # new id of every old page, V plane kept at +numPages
    pool2 = torch.empty_like(d_dev["pool"])
    pool2[mapping] = d_dev["pool"]
    d2 = dict(d_dev, pool=pool2, page_table=mapping[d_dev["page_table"].long()].int())
    out2, _ = _gpu_attention(d2, lists_dev, cfg, 0.08, ws)
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))


def test_sparse_decode_status_word_reports_bad_entries():
    """A list entry past the sequence's length and a page id outside the pool
    are skipped without a fault, and the optional status word says so (bit 2,
    bit 1); the output equals the oracle's on the list with those entries
    dropped.  Clean inputs leave the word at zero."""
    cfg = syn.DECODE_PARITY
    d = syn.make_decode(cfg)
    d_np = {k: (v.numpy() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    ctx = d_np["ctx"]
    rng = np.random.default_rng(5)
    lists = np.full((cfg.B, cfg.topK), -1, np.int32)
    for b, L in enumerate(ctx):
        n = min(int(L), 300)
        lists[b, :n] = np.sort(rng.choice(int(L), size=n, replace=False))
    d_dev = _to_dev(d)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    po, ps, pc = qb.sparse_decode_workspace_elems(cfg.B, cfg.Hkv, cfg.D)

    def run(lst, pt):
        ws = (torch.zeros(po, dtype=torch.float32, device=DEV), torch.zeros(ps, dtype=torch.float32, device=DEV),
              torch.zeros(pc, dtype=torch.int32, device=DEV))
        out = torch.full((cfg.B, 1, cfg.Hq, cfg.D), float("nan"), dtype=torch.float16, device=DEV)
        qb.sparse_decode(d_dev["q"], d_dev["pool"], pt, torch.from_numpy(lst[:, None, :].copy()).to(DEV),
                         d_dev["ctx"], out, *ws, D=cfg.D, scale=f32(cfg.scale), status=status)
        torch.cuda.synchronize()
        return to_np(out)[:, 0]

    run(lists, d_dev["page_table"])
    assert int(status.item()) == 0, "clean inputs set status bits"
    b_idx, b_page = 3, 5  # L = 2048 and 6000
    bad = lists.copy()
    bad[b_idx, 7] = int(ctx[b_idx]) + 11  # past the live length
    bad[b_idx, 9] = -5                    # negative, not the -1 padding
    pt_bad = d_np["page_table"].copy()
    page = int(lists[b_page, 0]) // TPP
    pt_bad[b_page, 0, page] = int(d["num_pages"]) * 2 + 3  # K page id outside the pool
    got = run(bad, torch.from_numpy(pt_bad).to(DEV))
    assert int(status.item()) == 6, f"status {int(status.item())} != bit 1 | bit 2"
    want_list = lists.copy()
    want_list[b_idx, 7] = -1
    want_list[b_idx, 9] = -1
    on_page = (want_list[b_page] >= 0) & (want_list[b_page] // TPP == page)
    assert on_page.sum() > 0
    want_list[b_page, on_page] = -1
    want = oracle.sparse_decode(d_np["q"][:, 0], d_np["pool"], d_np["page_table"], want_list, ctx, D=cfg.D,
                                scale=f32(cfg.scale))
    check_attention(got, want, "decode with bad entries dropped")
    assert qb.last_device_error(status) == 6  # the documented read of a device error word
