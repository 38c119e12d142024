"""Pins of the CPU oracle's indexer steps to things other than itself.

Each test checks one oracle function against a closed form, a hand-worked
fixture (tests/golden/), a library routine (numpy's float16 conversion) or
brute force, chosen so that a dropped term, a wrong sign or index, or a
transposed operand fails at least one of them.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest

from conftest import load_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ------------------------------------------------------------------ fp16 bits
def test_half_to_double_all_bit_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, oracle_mod.half_to_double(0x8000)) == -1.0


def test_double_to_half_matches_numpy_rne(oracle_mod):
    rng = np.random.default_rng(3)
    xs = [0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e9, 6.0e-8, 2.0 ** -24, 2.0 ** -25,
          2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -11)]
    # every midpoint between adjacent finite halves (exact ties) and neighbours
    h = np.arange(0, 0x7C00, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    h2 = (np.arange(0, 0x7C00, 37, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    mids = (h + h2) / 2
    xs += list(mids) + list(-mids) + list(np.nextafter(mids, 0)) + list(np.nextafter(mids, 1e9))
    xs += list(rng.normal(size=2000) * 10.0 ** rng.integers(-9, 5, size=2000))
    for x in xs:
        want = np.array([x], np.float64).astype(np.float16).view(np.uint16)[0]
        assert oracle_mod.double_to_half(x) == want, x
    assert oracle_mod.double_to_half(float("nan")) & 0x7C00 == 0x7C00


# --------------------------------------------------------------- RMSNorm*(1+w)
def test_rmsnorm_golden(oracle_mod):
    g = load_golden("rmsnorm.txt")
    x = np.array(g["x"], np.float16)
    for c in ("case1", "case2"):
        y = oracle_mod.index_q(x, np.array(g[f"{c}_w"], np.float32), rot=0, pos=0, theta=1e4, eps=0.0)
        np.testing.assert_allclose(y, g[f"{c}_y"], rtol=0, atol=1e-15)


def test_rmsnorm_closed_form_w0(oracle_mod):
    rng = np.random.default_rng(0)
    for di, eps in ((64, 1e-6), (128, 1e-6), (128, 0.5)):
        x = rng.normal(size=di).astype(np.float16)
        y = oracle_mod.index_q(x, np.zeros(di, np.float32), rot=0, pos=0, theta=1e4, eps=eps)
        ms = np.mean(x.astype(np.float64) ** 2)
        assert abs(np.sum(y * y) - di * ms / (ms + eps)) < 1e-12 * di
        # direction is x's
        np.testing.assert_allclose(y / x.astype(np.float64), 1 / np.sqrt(ms + eps), rtol=1e-14)


def test_rmsnorm_weight_is_one_plus_w(oracle_mod):
    rng = np.random.default_rng(1)
    x = rng.normal(size=64).astype(np.float16)
    w = rng.normal(scale=0.1, size=64).astype(np.float32)
    y0 = oracle_mod.index_q(x, np.zeros(64, np.float32), rot=0, pos=0, theta=1e4, eps=1e-6)
    y = oracle_mod.index_q(x, w, rot=0, pos=0, theta=1e4, eps=1e-6)
    np.testing.assert_allclose(y, y0 * (1.0 + w.astype(np.float64)), rtol=1e-14)


# ------------------------------------------------------------------ partial RoPE
def test_rope_golden_unit_vectors(oracle_mod):
    g = load_golden("rope.txt")
    di, rot, theta = g["di"][0], g["rot"][0], float(g["theta"][0])
    for c in ("case1", "case2", "case3", "case4"):
        # a unit vector survives RMSNorm as sqrt(di) * e (w = 0, eps = 0): undo that scale
        x = np.zeros(di, np.float16)
        x[g[f"{c}_in_dim"][0]] = 1.0
        y = oracle_mod.index_q(x, np.zeros(di, np.float32), rot=rot, pos=g[f"{c}_pos"][0], theta=theta,
                               eps=0.0) / math.sqrt(di)
        np.testing.assert_allclose(y, g[f"{c}_out"], rtol=0, atol=1e-12)


def _normed(oracle_mod, x, eps=1e-6):
    return oracle_mod.index_q(x, np.zeros(len(x), np.float32), rot=0, pos=0, theta=1e4, eps=eps)


def test_rope_is_complex_rotation(oracle_mod):
    """RoFormer's definition: pair j as a complex number times exp(i pos theta^(-2j/rot))."""
    rng = np.random.default_rng(2)
    for di, rot, pos in ((64, 32, 0), (64, 32, 7), (128, 64, 1234), (128, 128, 524287), (128, 64, 524284)):
        x = rng.normal(size=di).astype(np.float16)
        y = oracle_mod.index_q(x, np.zeros(di, np.float32), rot=rot, pos=pos, theta=1e4, eps=1e-6)
        n = _normed(oracle_mod, x)
        half = rot // 2
        z = n[:half] + 1j * n[half:rot]
        ang = pos * (1e4 ** (-2.0 * np.arange(half) / rot))
        zr = z * np.exp(1j * ang)
        # an f64 angle pos * inv_freq carries ~1 ulp of pos * inv_freq: the bound grows with pos
        atol = 1e-12 + 1e-15 * pos
        np.testing.assert_allclose(y[:half], zr.real, rtol=0, atol=atol)
        np.testing.assert_allclose(y[half:rot], zr.imag, rtol=0, atol=atol)
        np.testing.assert_array_equal(y[rot:], n[rot:])


def test_rope_relative_position_property(oracle_mod):
    """<R(a, m), R(b, n)> depends only on m - n."""
    rng = np.random.default_rng(4)
    a = rng.normal(size=128).astype(np.float16)
    b = rng.normal(size=128).astype(np.float16)
    w = np.zeros(128, np.float32)

    def dot(m, n):
        return np.dot(oracle_mod.index_q(a, w, 64, m, 1e4, 1e-6), oracle_mod.index_q(b, w, 64, n, 1e4, 1e-6))

    ref = dot(100, 37)
    for shift in (1, 1000, 400000):
        assert abs(dot(100 + shift, 37 + shift) - ref) < 1e-9
    assert abs(dot(101, 37) - ref) > 1e-6  # and it does depend on m - n


def test_rope_pos0_identity_and_norm_preserving(oracle_mod):
    rng = np.random.default_rng(5)
    x = rng.normal(size=128).astype(np.float16)
    n = _normed(oracle_mod, x)
    y0 = oracle_mod.index_q(x, np.zeros(128, np.float32), 64, 0, 1e4, 1e-6)
    np.testing.assert_array_equal(y0, n)
    y = oracle_mod.index_q(x, np.zeros(128, np.float32), 64, 9999, 1e4, 1e-6)
    for i in range(32):
        assert abs(math.hypot(y[i], y[i + 32]) - math.hypot(n[i], n[i + 32])) < 1e-12


# ------------------------------------------------------------------ block key
def test_block_key_is_mean_then_norm_then_rope(oracle_mod):
    rng = np.random.default_rng(6)
    di, rot = 64, 32
    # small integers: the mean of four rows is exact in fp16
    raw = rng.integers(-3, 4, size=(4, di)).astype(np.float16)
    raw[0] += (4 - raw.sum(axis=0) % 4) % 4  # make each column sum divisible by 4
    mean = (raw.astype(np.float64).sum(axis=0) / 4).astype(np.float16)
    w = rng.normal(scale=0.1, size=di).astype(np.float32)
    eps = 0.5  # a large eps makes a dropped 1/r visible through the norm
    for pos in (0, 4, 4096):
        kb, y64 = oracle_mod.block_key(raw, w, rot, pos, 1e4, eps)
        want = oracle_mod.index_q(mean, w, rot, pos, 1e4, eps)
        np.testing.assert_allclose(y64, want, rtol=0, atol=1e-13)
        # storage rounding is numpy's float16 RNE of the f64 value
        np.testing.assert_array_equal(kb.view(np.uint16), y64.astype(np.float16).view(np.uint16))


def test_block_key_identical_rows(oracle_mod):
    rng = np.random.default_rng(7)
    x = rng.normal(size=128).astype(np.float16)
    w = rng.normal(scale=0.1, size=128).astype(np.float32)
    kb, y64 = oracle_mod.block_key(np.stack([x] * 4), w, 64, 8, 1e4, 1e-6)
    np.testing.assert_allclose(y64, oracle_mod.index_q(x, w, 64, 8, 1e4, 1e-6), rtol=0, atol=1e-13)


# ---------------------------------------------------------------------- score
def test_score_golden(oracle_mod):
    g = load_golden("score.txt")
    q = np.array([g["q0"], g["q1"]], np.float64)
    for c in ("case1", "case2", "case3", "case4"):
        s = oracle_mod.block_score(q, np.array(g[f"{c}_k"], np.float16))
        assert s == pytest.approx(g[f"{c}_score"][0], abs=1e-15)


def test_score_relu_per_head_not_of_sum(oracle_mod):
    q = np.array([[1.0, 0, 0, 0], [-1.0, 0, 0, 0]])
    # relu of each head's dot: 1 + 0, while relu of the head sum would be 0
    assert oracle_mod.block_score(q, np.array([1, 0, 0, 0], np.float16)) == pytest.approx(0.5)


# --------------------------------------------------------------------- select
def _brute_top(scores, beta):
    n = len(scores)
    if n <= beta:
        return list(range(n))
    found = []
    for comb in itertools.combinations(range(n), beta):
        s = set(comb)
        ok = all((scores[g] > scores[h]) or (scores[g] == scores[h] and g < h)
                 for g in s for h in range(n) if h not in s)
        if ok:
            found.append(sorted(comb))
    assert len(found) == 1
    return found[0]


def test_select_equals_brute_force_with_ties(oracle_mod):
    rng = np.random.default_rng(8)
    for trial in range(300):
        n = int(rng.integers(0, 11))
        beta = int(rng.integers(1, 6))
        scores = rng.integers(0, 4, size=n).astype(np.float64)  # many exact ties
        if trial % 3 == 0:
            scores = rng.normal(size=n)
        got = list(oracle_mod.select(scores, beta))
        assert got == _brute_top(list(scores), beta), (scores, beta)


def test_select_all_zero_scores_take_lowest_ids(oracle_mod):
    assert list(oracle_mod.select(np.zeros(100), 7)) == list(range(7))


# --------------------------------------------------------------------- expand
def test_expand_golden(oracle_mod):
    g = load_golden("expand.txt")
    r, topK = g["ratio"][0], g["topK"][0]
    for c in ("case1", "case2", "case3"):
        t = g[f"{c}_t"][0]
        n_c = (t + 1) // r
        got = oracle_mod.expand(np.array(g[f"{c}_sel"], np.int32), n_c, t, r, topK)
        assert list(got) == g[f"{c}_list"]


def test_expand_invariants(oracle_mod):
    rng = np.random.default_rng(9)
    r, beta = 4, 8
    topK = beta * r + r - 1
    for _ in range(500):
        t = int(rng.integers(0, 400))
        n_c = (t + 1) // r
        k = min(n_c, beta)
        sel = np.sort(rng.choice(n_c, size=k, replace=False)) if k else np.zeros(0, np.int32)
        lst = oracle_mod.expand(sel.astype(np.int32), n_c, t, r, topK)
        valid = lst[lst >= 0]
        n = len(valid)
        assert np.all(lst[n:] == -1)                       # -1 only on the right
        assert len(np.unique(valid)) == n                  # distinct
        assert np.all(valid <= t)                          # causal
        assert n == k * r + (t + 1 - n_c * r)              # cnt(t)
        if n_c <= beta:
            assert list(valid) == list(range(t + 1))       # dense special case
