"""Seeded synthetic inputs for the QSA hot path.

Shared by the tests, the smoke check and the benchmark; both the CUDA path and
the CPU oracle receive the tensors made here.  This module holds none of the
method's arithmetic: only random values, lengths, page tables and layouts.

Workloads follow the five benchmark configurations of the QSA pages'
benchmark plan (prefill tiny / 8K / ragged batch, decode / long decode) plus
smaller parity shapes.  Values are N(0, 1) fp16, norm weights N(0, 0.1) fp32;
rows at or past a sequence's live length are poisoned with NaN so that any
read of them shows up in the outputs.
"""
from __future__ import annotations

import dataclasses
import math

import torch

TOKENS_PER_PAGE = 128


@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    Hi: int
    di: int
    rot: int
    ratio: int
    budget: int
    theta: float = 1.0e4
    eps: float = 1.0e-6
    ctx_lo: int | None = None  # None: every sequence is full length
    ctx_hi: int | None = None
    seed: int = 0

    @property
    def topK(self) -> int:
        return self.budget * self.ratio + self.ratio - 1

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    Hi: int
    di: int
    rot: int
    ratio: int
    budget: int
    ctx_lo: int
    ctx_hi: int
    max_ctx: int  # page-table capacity in tokens
    theta: float = 1.0e4
    eps: float = 1.0e-6
    seed: int = 0
    ctx_list: tuple | None = None  # explicit lengths (overrides ctx_lo/ctx_hi)

    @property
    def topK(self) -> int:
        return self.budget * self.ratio + self.ratio - 1

    @property
    def poolHeadDim(self) -> int:
        return self.D + self.di

    @property
    def maxPagesPerSeq(self) -> int:
        return -(-self.max_ctx // TOKENS_PER_PAGE)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


# The five benchmark workloads (seed 1000 + position in the list, from 1).
PREFILL_TINY = PrefillConfig("prefill_tiny_S512", B=1, S=512, Hq=8, Hkv=2, D=128, Hi=4, di=64, rot=32,
                             ratio=4, budget=16, seed=1001)
PREFILL_8K = PrefillConfig("prefill_S8192", B=1, S=8192, Hq=32, Hkv=4, D=128, Hi=8, di=128, rot=64,
                           ratio=4, budget=512, seed=1002)
PREFILL_RAGGED = PrefillConfig("prefill_ragged_B4_S16384", B=4, S=16384, Hq=32, Hkv=4, D=128, Hi=8,
                               di=128, rot=64, ratio=4, budget=512, ctx_lo=4096, ctx_hi=16384, seed=1003)
DECODE_32 = DecodeConfig("decode_B32_L2k-64k", B=32, Hq=32, Hkv=4, D=128, Hi=8, di=128, rot=64, ratio=4,
                         budget=512, ctx_lo=2048, ctx_hi=65536, max_ctx=65536, seed=1004)
DECODE_LONG = DecodeConfig("decode_long_B8_L512k", B=8, Hq=64, Hkv=8, D=128, Hi=8, di=128, rot=64, ratio=4,
                           budget=512, ctx_lo=524288, ctx_hi=524288, max_ctx=524288, seed=1005)
BENCH_CONFIGS = (PREFILL_TINY, PREFILL_8K, PREFILL_RAGGED, DECODE_32, DECODE_LONG)

# Prefill past 16K rows: the 28K prefill the qsa.rs page times (doc comment of
# qsa_score_rows_tc), 64K, and a ragged batch whose rows see up to 5000 blocks.
PREFILL_28K = PrefillConfig("prefill_S28672", B=1, S=28672, Hq=32, Hkv=4, D=128, Hi=8, di=128, rot=64,
                            ratio=4, budget=512, seed=28)
PREFILL_64K = PrefillConfig("prefill_S65536", B=1, S=65536, Hq=32, Hkv=4, D=128, Hi=8, di=128, rot=64,
                            ratio=4, budget=512, seed=64)
PREFILL_LONG_RAGGED = PrefillConfig("prefill_ragged_B2_S20000", B=2, S=20000, Hq=32, Hkv=4, D=128, Hi=8,
                                    di=128, rot=64, ratio=4, budget=512, ctx_lo=12000, ctx_hi=20000, seed=20)

# Smaller shapes for element-by-element parity (several tiles and a ragged tail).
PREFILL_PARITY = PrefillConfig("prefill_parity", B=2, S=3001, Hq=16, Hkv=2, D=128, Hi=8, di=128, rot=64,
                               ratio=4, budget=128, ctx_lo=1500, ctx_hi=3001, seed=7)
DECODE_PARITY = DecodeConfig("decode_parity", B=6, Hq=16, Hkv=2, D=128, Hi=8, di=128, rot=64, ratio=4,
                             budget=128, ctx_lo=1, ctx_hi=6000, max_ctx=6144, seed=11,
                             ctx_list=(1, 4, 515, 2048, 4099, 6000))


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_fp16(shape, g, device="cpu"):
    return torch.randn(shape, generator=g, dtype=torch.float32, device=device).to(torch.float16)


def context_lengths(cfg, g=None) -> torch.Tensor:
    """int32 [B] live lengths of a config, drawn with its seed."""
    if getattr(cfg, "ctx_list", None):
        return torch.tensor(cfg.ctx_list, dtype=torch.int32)
    if g is None:
        g = _gen(cfg.seed + 1)
    if cfg.ctx_lo is None:
        return torch.full((cfg.B,), cfg.S, dtype=torch.int32)
    return torch.randint(cfg.ctx_lo, cfg.ctx_hi + 1, (cfg.B,), generator=g, dtype=torch.int64).to(torch.int32)


def make_prefill(cfg: PrefillConfig, poison: bool = True) -> dict:
    """CPU tensors of one prefill batch: q/k/v, idxQ/idxK, norm weights, lengths."""
    g = _gen(cfg.seed)
    ctx = context_lengths(cfg)
    B, S = cfg.B, cfg.S
    t = {
        "q": _normal_fp16((B, S, cfg.Hq, cfg.D), g),
        "k": _normal_fp16((B, S, cfg.Hkv, cfg.D), g),
        "v": _normal_fp16((B, S, cfg.Hkv, cfg.D), g),
        "idxQ": _normal_fp16((B, S, cfg.Hi, cfg.di), g),
        "idxK": _normal_fp16((B, S, cfg.di), g),
        "wq": (0.1 * torch.randn((cfg.di,), generator=g)).to(torch.float32),
        "wk": (0.1 * torch.randn((cfg.di,), generator=g)).to(torch.float32),
        "ctx": ctx,
    }
    if poison:
        for b in range(B):
            L = int(ctx[b])
            for name in ("q", "k", "v", "idxQ", "idxK"):
                t[name][b, L:] = float("nan")
    return t


def make_decode(cfg: DecodeConfig, device="cpu") -> dict:
    """One decode step: pool, page table, new-token q/idxQ/idxK, weights, lengths.

    The pool holds 2*numPages pages: K pages are a random permutation of
    [0, numPages) over every used page of every sequence, and each V page id is
    its K page id + numPages.  The whole pool, tails included, is N(0, 1) fp16
    (a well-formed synthetic indexer state).  With device="cuda" the pool is
    drawn on the GPU (large pools); everything else is drawn on the CPU.
    """
    g = _gen(cfg.seed)
    ctx = context_lengths(cfg, _gen(cfg.seed + 1))
    B = cfg.B
    pages_per_seq = [-(-int(L) // TOKENS_PER_PAGE) for L in ctx]
    num_pages = max(1, sum(pages_per_seq))
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    page_table = torch.zeros((B, 2, cfg.maxPagesPerSeq), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per_seq):
        page_table[b, 0, :n] = perm[off:off + n]
        page_table[b, 1, :n] = perm[off:off + n] + num_pages
        off += n
    shape = (2 * num_pages, TOKENS_PER_PAGE, cfg.Hkv, cfg.poolHeadDim)
    if str(device).startswith("cuda"):
        gd = _gen(cfg.seed + 2, device=device)
        pool = torch.randn(shape, generator=gd, dtype=torch.float16, device=device)
    else:
        pool = _normal_fp16(shape, _gen(cfg.seed + 2))
    return {
        "pool": pool,
        "page_table": page_table,
        "q": _normal_fp16((B, 1, cfg.Hq, cfg.D), g),
        "idxQ": _normal_fp16((B, cfg.Hi, cfg.di), g),
        "idxK": _normal_fp16((B, cfg.di), g),
        "wq": (0.1 * torch.randn((cfg.di,), generator=g)).to(torch.float32),
        "wk": (0.1 * torch.randn((cfg.di,), generator=g)).to(torch.float32),
        "ctx": ctx,
        "num_pages": num_pages,
    }


def random_lists(B: int, S: int, topK: int, ctx, seed: int, fill: float = 1.0,
                 causal: bool = True) -> torch.Tensor:
    """Valid index lists for attention-only tests: distinct live token ids,
    -1 padded on the right, in random order.  Row t draws from [0, t] when
    `causal`, else from [0, L); about `fill` of the width is used."""
    g = _gen(seed)
    out = torch.full((B, S, topK), -1, dtype=torch.int32)
    for b in range(B):
        L = int(ctx[b])
        for t in range(L):
            span = t + 1 if causal else L
            n = min(span, max(1, int(round(fill * topK))))
            pick = torch.randperm(span, generator=g)[:n].to(torch.int32)
            out[b, t, :n] = pick
    return out


def qsa_like_lists(B: int, S: int, ctx, ratio: int, budget: int, topK: int, seed: int,
                   device="cpu", chunk_rows: int = 1024) -> torch.Tensor:
    """Index lists with the indexer's structure but a random block choice.

    Row t < L keeps every complete block when n_c(t) <= budget, else `budget`
    complete blocks drawn uniformly; the blocks expand to their `ratio` tokens
    and the causal tail follows; ascending, -1 padded.  Rows t >= L are -1.
    For attention inputs at sizes where a CPU reference selection is slow."""
    g = _gen(seed, device=device)
    out = torch.full((B, S, topK), -1, dtype=torch.int32, device=device)
    nbmax = max(S // ratio, 1)
    big = 1 << 30
    for b in range(B):
        L = int(ctx[b])
        for r0 in range(0, L, chunk_rows):
            r1 = min(L, r0 + chunk_rows)
            t = torch.arange(r0, r1, device=device)
            n_c = (t + 1) // ratio
            blk = torch.arange(nbmax, device=device)
            valid = blk[None, :] < n_c[:, None]
            key = torch.rand((r1 - r0, nbmax), generator=g, device=device)
            key = torch.where(valid, key, torch.full_like(key, -1.0))
            k = min(budget, nbmax)
            top = torch.topk(key, k, dim=1).indices
            chosen = torch.zeros_like(valid)
            chosen.scatter_(1, top, True)
            chosen &= valid
            tok = torch.arange(S, device=device)
            tmask = chosen.repeat_interleave(ratio, dim=1)
            if tmask.shape[1] < S:
                tmask = torch.cat([tmask, torch.zeros((r1 - r0, S - tmask.shape[1]), dtype=torch.bool,
                                                      device=device)], dim=1)
            tmask = tmask[:, :S] | ((tok[None, :] >= (n_c * ratio)[:, None]) & (tok[None, :] <= t[:, None]))
            keyed = torch.where(tmask, tok[None, :].expand(r1 - r0, S), torch.full((1, 1), big, device=device))
            srt = torch.sort(keyed, dim=1).values[:, :topK]
            srt = torch.where(srt == big, torch.full_like(srt, -1), srt)
            if srt.shape[1] < topK:
                srt = torch.cat([srt, torch.full((r1 - r0, topK - srt.shape[1]), -1, device=device,
                                                 dtype=srt.dtype)], dim=1)
            out[b, r0:r1] = srt.to(torch.int32)
    return out
