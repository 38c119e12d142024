"""Helpers shared by the GPU parity tests: running the CUDA path through the
binding, reading its outputs back, and the comparisons the parity bar uses.

Selection parity (the benchmark spec's tolerance): a row's GPU block set must equal
the oracle's, except for swaps at the top-k cut where the oracle's scores tie
within 1e-6 relative -- every block in the symmetric difference must score
within 1e-6 * c of the oracle's budget-th largest score, with
c = max(|cut|, row max).  Attention parity: max |gpu - oracle_f64| <= 2e-3 on
live rows, exact fp16 zeros on padded rows, no NaN anywhere.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from block_sparse_gqa_qsa_gb300 import _binding as qb

ATTN_ATOL = 2e-3
TIE_REL = 1e-6


def f32(x) -> float:
    """The value as the fp32 the C ABI receives (so both sides use one constant)."""
    return float(np.float32(x))


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


# ------------------------------------------------------------ CUDA path runs
def gpu_indexer_prefill(t: dict, cfg, dev="cuda", topK=None, budget=None):
    """Runs qsa_indexer_prefill; returns (indices [B,S,topK] device, workspace)."""
    topK = topK or cfg.topK
    budget = budget or cfg.budget
    B, S = cfg.B, cfg.S
    ws = qb.alloc_workspace(qb.indexer_prefill_workspace_size(B, S, cfg.di, cfg.ratio), dev)
    ind = torch.full((B, S, topK), 7, dtype=torch.int32, device=dev)  # garbage: every slot must be written
    qb.indexer_prefill(t["idxQ"], t["idxK"], t["wq"], t["wk"], t["ctx"], ind, ws, rot=cfg.rot, ratio=cfg.ratio,
                       budget=budget, topK=topK, theta=cfg.theta, eps=cfg.eps)
    return ind, ws


def workspace_kbar(ws: torch.Tensor, B: int, S: int, di: int, ratio: int) -> np.ndarray:
    """Block keys the prefill indexer left in its workspace (fp16 [B, S/r, di] after a 256-byte head)."""
    nb = S // ratio
    raw = ws[256:256 + B * nb * di * 2]
    return to_np(raw).view(np.float16).reshape(B, nb, di)


def same_fp16_bits(a: np.ndarray, b: np.ndarray) -> bool:
    """fp16 arrays equal bit for bit, except that an exact zero may carry either sign.

    Both sides round the same exact value once; a component whose exact value
    is 0 gets its sign from IEEE sign-of-zero rules, which depend on operation
    order (0*cos - 0*sin is -0 in f64 when cos < 0), so the sign is no claim.
    """
    ab, bb = a.view(np.uint16), b.view(np.uint16)
    zero = ((ab & 0x7FFF) == 0) & ((bb & 0x7FFF) == 0)
    return bool(np.all((ab == bb) | zero))


def oracle_prefill_lists(t_np: dict, cfg, rows=None, want_scores=False, budget=None, topK=None):
    return oracle.indexer_prefill(t_np["idxQ"], t_np["idxK"], t_np["wq"], t_np["wk"], t_np["ctx"], rot=cfg.rot,
                                  ratio=cfg.ratio, budget=budget or cfg.budget, topK=topK or cfg.topK,
                                  theta=cfg.theta, eps=f32(cfg.eps), rows=rows, want_scores=want_scores,
                                  want_kbar=False)


# ------------------------------------------------------------ comparisons
def list_blocks(lst: np.ndarray, t: int, ratio: int):
    v = lst[lst >= 0]
    n_c = (t + 1) // ratio
    return set(int(j) // ratio for j in v if j < n_c * ratio)


def check_list(lst: np.ndarray, t: int, L: int, ratio: int, budget: int) -> None:
    """Index-list contract of one row: distinct, 0 <= j <= t, -1 only on the
    right, whole blocks plus the whole causal tail, count = cnt(t)."""
    if t >= L:
        assert np.all(lst == -1), f"row {t} >= L={L} not all -1"
        return
    n = int(np.sum(lst >= 0))
    assert np.all(lst[:n] >= 0) and np.all(lst[n:] == -1), f"row {t}: -1 not only on the right"
    v = lst[:n]
    assert len(np.unique(v)) == n, f"row {t}: duplicates"
    assert v.min() >= 0 and v.max() <= t, f"row {t}: index outside [0, t]"
    n_c = (t + 1) // ratio
    assert n == min(n_c, budget) * ratio + (t + 1 - n_c * ratio), f"row {t}: count {n}"
    s = set(v.tolist())
    assert set(range(n_c * ratio, t + 1)) <= s, f"row {t}: tail incomplete"
    blocks = {j // ratio for j in s if j < n_c * ratio}
    assert len(blocks) * ratio + (t + 1 - n_c * ratio) == n, f"row {t}: partial block"


def check_lists_device(ind: torch.Tensor, ctx, ratio: int, budget: int) -> None:
    """Vectorised structure checks of every row of [B,S,topK] lists (ascending emission)."""
    B, S, topK = ind.shape
    dev = ind.device
    t = torch.arange(S, device=dev)
    for b in range(B):
        L = int(ctx[b])
        x = ind[b].long()
        assert bool((x[L:] == -1).all()), "padded rows must be all -1"
        x = x[:L]
        if L == 0:
            continue
        tt = t[:L]
        n_c = (tt + 1) // ratio
        cnt = torch.clamp(n_c, max=budget) * ratio + (tt + 1 - n_c * ratio)
        valid = x >= 0
        assert bool((valid.sum(1) == cnt).all()), "count != cnt(t)"
        pos = torch.arange(topK, device=dev)
        assert bool((valid == (pos[None, :] < cnt[:, None])).all()), "-1 only on the right"
        big = torch.where(valid, x, torch.full_like(x, 1 << 40))
        assert bool((big[:, 1:] > big[:, :-1])[valid[:, 1:]].all()), "lists must be strictly ascending"
        assert bool((torch.where(valid, x, torch.zeros_like(x)) <= tt[:, None]).all()), "index > t"
        nsel = torch.clamp(n_c, max=budget)
        # block part: groups of `ratio` consecutive tokens starting at a multiple of ratio
        head = pos[None, :] < (nsel * ratio)[:, None]
        grp0 = torch.gather(x, 1, (pos - pos % ratio)[None, :].expand(L, topK))
        ok = (x == grp0 + (pos % ratio)[None, :]) & (grp0 % ratio == 0) & (x < (n_c * ratio)[:, None])
        assert bool(ok[head].all()), "block part malformed"
        tail = valid & ~head
        want = (n_c * ratio)[:, None] + (pos[None, :] - (nsel * ratio)[:, None])
        assert bool((x == want)[tail].all()), "tail malformed"


def compare_selection(gpu_row: np.ndarray, ora_row: np.ndarray, scores: np.ndarray, t: int, ratio: int,
                      budget: int) -> bool:
    """True when the block sets are equal; raises when they differ beyond the tie tolerance."""
    gb, ob = list_blocks(gpu_row, t, ratio), list_blocks(ora_row, t, ratio)
    if gb == ob:
        return True
    n_c = (t + 1) // ratio
    s = scores[:n_c]
    assert len(gb) == len(ob), f"row {t}: {len(gb)} vs {len(ob)} blocks"
    cut = np.sort(s)[::-1][budget - 1]
    c = max(abs(cut), float(s.max()))
    diff = sorted(gb ^ ob)
    worst = max(abs(s[g] - cut) for g in diff)
    assert worst <= TIE_REL * c, f"row {t}: blocks {diff[:6]} differ by {worst:.3e} > {TIE_REL} * {c:.3f}"
    return False


def check_attention(gpu: np.ndarray, ref: np.ndarray, what: str) -> float:
    g = gpu.astype(np.float64)
    assert not np.isnan(g).any(), f"{what}: NaN in output"
    err = float(np.max(np.abs(g - ref))) if g.size else 0.0
    assert err <= ATTN_ATOL, f"{what}: max abs error {err:.3e} > {ATTN_ATOL}"
    return err
