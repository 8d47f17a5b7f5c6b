"""Pins for the oracle's ring-step merge and for the whole chunked method.

The pages' central claim is that ring, Ulysses and unified attention give the same output as
unsplit attention (diffusers PR #12693: "identical output" across backends; HF docs "Context
parallelism", Ring Attention: after one loop every rank has seen every token's K/V).  So the
chunked-and-merged oracle must equal the unsplit oracle to fp64 rounding for every split."""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle

RNG = np.random.default_rng(99)


def rand(*shape):
    return RNG.standard_normal(shape)


def test_merge_lse_is_logsumexp():
    """Merging partials over disjoint key sets: lse = logsumexp of the partial lses (scipy)."""
    l = rand(6, 5) * 4
    o = rand(6, 5, 3)
    run_o, run_l = o[0], l[0]
    for i in range(1, 6):
        run_o, run_l = oracle.merge(run_o, run_l, o[i], l[i])
    assert np.allclose(run_l, logsumexp(l, axis=0), atol=1e-12)
    w = np.exp(l - logsumexp(l, axis=0))
    assert np.allclose(run_o, (w[..., None] * o).sum(axis=0), atol=1e-12)


def test_merge_with_empty_partial():
    o, l = rand(4, 8), rand(4)
    z, zl = np.full((4, 8), 123.0), np.full(4, -math.inf)
    mo, ml = oracle.merge(o, l, z, zl)
    assert np.array_equal(mo, o) and np.array_equal(ml, l)
    mo, ml = oracle.merge(z, zl, o, l)
    assert np.array_equal(mo, o) and np.array_equal(ml, l)
    mo, ml = oracle.merge(np.zeros((4, 8)), zl, z, zl)
    assert np.all(ml == -math.inf) and np.all(mo == 0)


def test_merge_commutative_associative():
    o = rand(3, 10, 4)
    l = rand(3, 10) * 3
    ab, abl = oracle.merge(o[0], l[0], o[1], l[1])
    ba, bal = oracle.merge(o[1], l[1], o[0], l[0])
    assert np.allclose(ab, ba, atol=1e-13) and np.allclose(abl, bal, atol=1e-13)
    left = oracle.merge(ab, abl, o[2], l[2])
    bc, bcl = oracle.merge(o[1], l[1], o[2], l[2])
    right = oracle.merge(o[0], l[0], bc, bcl)
    assert np.allclose(left[0], right[0], atol=1e-13) and np.allclose(left[1], right[1], atol=1e-13)


def test_merge_extreme_lse_gap():
    o1, o2 = rand(2, 4), rand(2, 4)
    mo, ml = oracle.merge(o1, np.array([0.0, 800.0]), o2, np.array([800.0, 0.0]))
    assert np.allclose(mo[0], o2[0]) and np.allclose(mo[1], o1[1])
    assert np.allclose(ml, [800.0, 800.0])


def test_two_chunk_split_by_hand():
    """Split keys into two halves, attend to each, merge: equals attention over all keys."""
    S, D = 29, 8
    q, k, v = rand(1, S, 2, D), rand(1, S, 2, D), rand(1, S, 2, D)
    full_o, full_l = oracle.attention(q, k, v, 0.35)
    a_o, a_l = oracle.attention(q, k[:, :11], v[:, :11], 0.35)
    b_o, b_l = oracle.attention(q, k[:, 11:], v[:, 11:], 0.35)
    mo, ml = oracle.merge(a_o, a_l, b_o, b_l)
    assert np.allclose(mo, full_o, atol=1e-12) and np.allclose(ml, full_l, atol=1e-12)


def _random_lens(total, parts, rng):
    cuts = np.sort(rng.choice(np.arange(1, total), size=parts - 1, replace=False)) if parts > 1 else []
    edges = [0, *cuts, total]
    return [int(edges[i + 1] - edges[i]) for i in range(parts)]


@pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("order", ["contiguous", "zigzag", "stripe"])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_equals_unsplit(R, order, causal):
    B, S, H, D = 1, 61, 2, 8
    q, k, v = rand(B, S, H, D), rand(B, S, H, D), rand(B, S, H, D)
    ref_o, ref_l = oracle.attention(q, k, v, 0.3, causal)
    o, l = oracle.usp_attention(q, k, v, 0.3, causal, 1, R, order)
    assert np.allclose(o, ref_o, rtol=1e-12, atol=1e-12)
    assert np.allclose(l, ref_l, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("U,R", [(2, 1), (3, 1), (4, 1), (2, 2), (3, 2), (2, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_unified_grid_equals_unsplit_uneven(U, R, causal):
    B, S, H, D = 2, 47, 5, 8     # S and H divisible by nothing useful: Ulysses Anything case
    q, k, v = rand(B, S, H, D), rand(B, S, H, D), rand(B, S, H, D)
    ref_o, ref_l = oracle.attention(q, k, v, 0.4, causal)
    rng = np.random.default_rng(U * 10 + R)
    ring_len = oracle.default_split(S, R)
    seq_lens = []
    for r in range(R):
        seq_lens += _random_lens(ring_len[r], U, rng)
    o, l = oracle.usp_attention(q, k, v, 0.4, causal, U, R, "contiguous", seq_lens)
    assert np.allclose(o, ref_o, rtol=1e-12, atol=1e-12)
    assert np.allclose(l, ref_l, rtol=1e-12, atol=1e-12)


def test_one_token_chunks():
    B, S, H, D = 1, 9, 3, 4
    q, k, v = rand(B, S, H, D), rand(B, S, H, D), rand(B, S, H, D)
    ref = oracle.attention(q, k, v, 0.5, True)
    o, l = oracle.usp_attention(q, k, v, 0.5, True, 1, 9, "contiguous")
    assert np.allclose(o, ref[0], atol=1e-12) and np.allclose(l, ref[1], atol=1e-12)
    o, l = oracle.usp_attention(q, k, v, 0.5, False, 3, 1, "contiguous", [1, 7, 1], [1, 1, 1])
    ref = oracle.attention(q, k, v, 0.5, False)
    assert np.allclose(o, ref[0], atol=1e-12) and np.allclose(l, ref[1], atol=1e-12)


def test_uneven_head_counts():
    B, S, H, D = 1, 12, 4, 4
    q, k, v = rand(B, S, H, D), rand(B, S, H, D), rand(B, S, H, D)
    ref = oracle.attention(q, k, v, 0.5, False)
    o, l = oracle.usp_attention(q, k, v, 0.5, False, 3, 1, "contiguous", [4, 4, 4], [2, 1, 1])
    assert np.allclose(o, ref[0], atol=1e-12) and np.allclose(l, ref[1], atol=1e-12)
