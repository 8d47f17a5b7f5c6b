"""Pins for the oracle's attention: brute force, torch's fp64 SDPA, closed forms and invariants.

None of these re-types the oracle's formula: brute force is pure-Python loops without the max
shift, torch's ``scaled_dot_product_attention`` is an independent library implementation, and
the closed forms follow from the definition by hand."""
import math

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def brute_force(q, k, v, scale, allowed):
    """Explicit sums over keys with math.fsum, no max shift (tiny inputs only)."""
    Sq, D = q.shape
    out = np.zeros((Sq, v.shape[1]))
    lse = np.full(Sq, -math.inf)
    for i in range(Sq):
        js = [j for j in range(k.shape[0]) if allowed[i][j]]
        if not js:
            continue
        e = {j: math.exp(scale * math.fsum(q[i, d] * k[j, d] for d in range(D))) for j in js}
        z = math.fsum(e.values())
        lse[i] = math.log(z)
        for d in range(v.shape[1]):
            out[i, d] = math.fsum(e[j] * v[j, d] for j in js) / z
    return out, lse


@pytest.mark.parametrize("Sq,Sk,D,causal", [(5, 7, 4, False), (9, 9, 8, True), (3, 11, 2, True),
                                            (1, 1, 3, False), (16, 5, 8, True)])
def test_brute_force_tiny(Sq, Sk, D, causal):
    q, k, v = rand(1, Sq, 1, D), rand(1, Sk, 1, D), rand(1, Sk, 1, D)
    scale = 1.0 / math.sqrt(D)
    qp = np.arange(Sq) + (Sk - Sq if Sk > Sq else 0)
    kp = np.arange(Sk)
    o, l = oracle.attention(q, k, v, scale, causal, qp, kp)
    allowed = [[(not causal) or kp[j] <= qp[i] for j in range(Sk)] for i in range(Sq)]
    bo, bl = brute_force(q[0, :, 0], k[0, :, 0], v[0, :, 0], scale, allowed)
    assert np.allclose(o[0, :, 0], bo, rtol=1e-12, atol=1e-12)
    assert np.allclose(l[0, :, 0], bl, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("B,S,H,D,causal", [(2, 37, 3, 16, False), (1, 64, 2, 64, True),
                                            (1, 130, 1, 128, True), (3, 20, 4, 8, False)])
def test_matches_torch_sdpa_fp64(B, S, H, D, causal):
    q, k, v = rand(B, S, H, D), rand(B, S, H, D), rand(B, S, H, D)
    scale = 1.0 / math.sqrt(D)
    o, _ = oracle.attention(q, k, v, scale, causal)
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    assert np.allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-12)


def test_matches_torch_sdpa_cross_length_mask():
    """Sq != Sk with global positions: the mask torch receives is built from positions."""
    Sq, Sk, D = 12, 40, 16
    q, k, v = rand(1, Sq, 2, D), rand(1, Sk, 2, D), rand(1, Sk, 2, D)
    qp = np.arange(20, 20 + Sq)
    kp = np.arange(Sk)
    o, _ = oracle.attention(q, k, v, 0.25, True, qp, kp)
    mask = torch.from_numpy(kp[None, :] <= qp[:, None])
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.25)
    assert np.allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-12)


def test_zero_query_closed_form():
    """Q = 0: every visible score is 0, so out = mean of the visible V rows and lse = ln |J|."""
    S, D = 23, 8
    q = np.zeros((1, S, 1, D))
    k, v = rand(1, S, 1, D), rand(1, S, 1, D)
    o, l = oracle.attention(q, k, v, 0.3, causal=True)
    for i in range(S):
        assert np.allclose(o[0, i, 0], v[0, : i + 1, 0].mean(axis=0), atol=1e-13)
        assert abs(l[0, i, 0] - math.log(i + 1)) < 1e-13


def test_constant_v_gives_v():
    S, D = 31, 16
    q, k = rand(2, S, 3, D, scale=3.0), rand(2, S, 3, D, scale=3.0)
    row = rand(D)
    v = np.broadcast_to(row, (2, S, 3, D)).copy()
    o, _ = oracle.attention(q, k, v, 1.0 / math.sqrt(D), causal=False)
    assert np.allclose(o, row, atol=1e-12)


def test_single_visible_key():
    """Causal row 0 sees only key 0: out = v_0, lse = scale q_0 . k_0."""
    D = 8
    q, k, v = rand(1, 5, 1, D), rand(1, 5, 1, D), rand(1, 5, 1, D)
    o, l = oracle.attention(q, k, v, 0.7, causal=True)
    assert np.allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-14)
    assert abs(l[0, 0, 0] - 0.7 * float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-13


def test_two_key_closed_form():
    """q = (1, 0), keys (1, 0) and (0, 1), scale 1: lse = ln(e + 1), out = (e v0 + v1) / (e + 1)."""
    q = np.array([1.0, 0.0]).reshape(1, 1, 1, 2)
    k = np.array([[1.0, 0.0], [0.0, 1.0]]).reshape(1, 2, 1, 2)
    v = np.array([[2.0, -1.0], [0.5, 4.0]]).reshape(1, 2, 1, 2)
    o, l = oracle.attention(q, k, v, 1.0)
    e = math.e
    assert abs(l[0, 0, 0] - math.log(e + 1.0)) < 1e-15
    assert np.allclose(o[0, 0, 0], (e * v[0, 0, 0] + v[0, 1, 0]) / (e + 1.0), atol=1e-15)


def test_lse_bounds_and_empty_rows():
    S, D = 40, 8
    q, k, v = rand(1, S, 1, D, scale=2), rand(1, S, 1, D, scale=2), rand(1, S, 1, D)
    qp = np.arange(S)
    kp = np.arange(S) + 10  # first 10 queries see nothing
    o, l = oracle.attention(q, k, v, 0.5, True, qp, kp)
    s = 0.5 * q[0, :, 0] @ k[0, :, 0].T
    for i in range(S):
        vis = kp <= qp[i]
        if not vis.any():
            assert l[0, i, 0] == -math.inf and np.all(o[0, i, 0] == 0)
            continue
        mx = s[i, vis].max()
        assert mx - 1e-12 <= l[0, i, 0] <= mx + math.log(vis.sum()) + 1e-12


def test_key_permutation_invariance():
    S, D = 33, 16
    q, k, v = rand(1, S, 2, D), rand(1, S, 2, D), rand(1, S, 2, D)
    perm = RNG.permutation(S)
    o1, l1 = oracle.attention(q, k, v, 0.25)
    o2, l2 = oracle.attention(q, k[:, perm], v[:, perm], 0.25)
    assert np.allclose(o1, o2, atol=1e-13) and np.allclose(l1, l2, atol=1e-13)


def test_attention_rows_matches_full():
    S, D = 50, 8
    q, k, v = rand(1, S, 1, D), rand(1, S, 1, D), rand(1, S, 1, D)
    o, l = oracle.attention(q, k, v, 0.3, causal=True)
    rows = np.array([0, 7, 49])
    ro, rl = oracle.attention_rows(q[0, rows, 0], k[0, :, 0], v[0, :, 0], 0.3, True, rows)
    assert np.allclose(ro, o[0, rows, 0], atol=1e-14) and np.allclose(rl, l[0, rows, 0], atol=1e-14)


def test_widen_bf16_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x4049, 0x7F80, 0x0001], dtype=np.uint16)
    x = oracle.widen_bf16(bits)
    assert x[0] == 1.0 and x[1] == -1.0 and x[2] == 0.0 and x[4] == math.inf
    assert x[3] == 3.140625
    assert x[5] == 2.0 ** -133  # smallest bf16 subnormal
