"""Planted mistakes in the oracle (on the CPU): every plausible error in its arithmetic must be
caught by at least one pin of the kind ``tests/test_oracle_*.py`` uses (pure-Python brute force
without a max shift, torch's fp64 SDPA, closed forms, invariants), while the real oracle passes all
of them.  This shows that the pins discriminate, not only that they pass."""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.usp as ousp

RNG = np.random.default_rng(77)
NEG_INF = float("-inf")


# ------------------------------------------------------------------------------------------------
# attention pins (independent of the oracle's formula)
# ------------------------------------------------------------------------------------------------

def _brute(q, k, v, scale, allowed):
    Sq, D = q.shape
    out = np.zeros((Sq, v.shape[1]))
    lse = np.full(Sq, NEG_INF)
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


def _pin_brute_force():
    Sq, Sk, D = 6, 9, 4
    q, k, v = (RNG.standard_normal((1, n, 1, D)) for n in (Sq, Sk, Sk))
    scale = 1.0 / math.sqrt(D)
    qp, kp = np.arange(Sq) + (Sk - Sq), np.arange(Sk)
    for causal in (False, True):
        o, l = oracle.attention(q, k, v, scale, causal, qp, kp)
        allowed = [[(not causal) or kp[j] <= qp[i] for j in range(Sk)] for i in range(Sq)]
        bo, bl = _brute(q[0, :, 0], k[0, :, 0], v[0, :, 0], scale, allowed)
        assert np.allclose(o[0, :, 0], bo, rtol=1e-12, atol=1e-12)
        assert np.allclose(l[0, :, 0], bl, rtol=1e-12, atol=1e-12)


def _pin_torch_sdpa():
    B, S, H, D = 1, 19, 2, 8
    q, k, v = (RNG.standard_normal((B, S, H, D)) for _ in range(3))
    scale = 1.0 / math.sqrt(D)
    for causal in (False, True):
        o, _ = oracle.attention(q, k, v, scale, causal)
        tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                               scale=scale)
        assert np.allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-12)


def _pin_zero_query():
    # Q = 0: every visible score is 0, so out = mean of the visible V rows and lse = ln |J|
    S, D = 7, 3
    q = np.zeros((1, S, 1, D))
    k, v = RNG.standard_normal((1, S, 1, D)), RNG.standard_normal((1, S, 1, D))
    o, l = oracle.attention(q, k, v, 0.5, True)
    for i in range(S):
        assert np.allclose(o[0, i, 0], v[0, :i + 1, 0].mean(axis=0), atol=1e-13)
        assert abs(l[0, i, 0] - math.log(i + 1)) < 1e-13


def _pin_single_key():
    # one visible key: out = its V row, lse = its scaled score
    D = 5
    q, k, v = (RNG.standard_normal((1, 1, 1, D)) for _ in range(3))
    o, l = oracle.attention(q, k, v, 0.3)
    assert np.allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-14)
    assert abs(l[0, 0, 0] - 0.3 * float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-13


ATTENTION_PINS = (_pin_brute_force, _pin_torch_sdpa, _pin_zero_query, _pin_single_key)


def _caught(pins) -> list[str]:
    failed = []
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    return failed


# ------------------------------------------------------------------------------------------------
# planted mistakes in the attention
# ------------------------------------------------------------------------------------------------

def _head_mutant(kind):
    def head(q, k, v, scale, allowed):
        Sq, D = q.shape[0], v.shape[1]
        if k.shape[0] == 0:
            return np.zeros((Sq, D)), np.full(Sq, NEG_INF)
        s = (q @ k.T) if kind == "scale dropped" else scale * (q @ k.T)
        if kind == "key index transposed" and s.shape[0] == s.shape[1]:
            s = s.T
        if allowed is not None and kind != "mask ignored":
            s = np.where(allowed, s, NEG_INF)
        m = s.max(axis=1)
        empty = ~np.isfinite(m)
        m_safe = np.where(empty, 0.0, m)
        w = np.exp((m_safe[:, None] - s) if kind == "exponent sign flipped" else (s - m_safe[:, None]))
        w = np.where(np.isfinite(w), w, 0.0)
        l = w.sum(axis=1)
        denom = np.where(empty, 1.0, l)[:, None]
        out = (w @ v) if kind == "no normalisation" else (w @ v) / denom
        if kind == "lse without the max":
            lse = np.log(np.where(empty, 1.0, l))
        elif kind == "lse in log2":
            lse = m_safe + np.log2(np.where(empty, 1.0, l))
        else:
            lse = m_safe + np.log(np.where(empty, 1.0, l))
        out[empty] = 0.0
        lse[empty] = NEG_INF
        return out, lse

    return head


HEAD_MUTANTS = ["scale dropped", "key index transposed", "mask ignored", "exponent sign flipped",
                "no normalisation", "lse without the max", "lse in log2"]


def test_real_oracle_passes_every_attention_pin():
    assert _caught(ATTENTION_PINS) == []


@pytest.mark.parametrize("kind", HEAD_MUTANTS)
def test_attention_mutant_is_caught(kind, monkeypatch):
    monkeypatch.setattr(ousp, "_attention_head", _head_mutant(kind))
    assert _caught(ATTENTION_PINS), f"no pin catches: {kind}"


def test_causal_mask_off_by_one_is_caught(monkeypatch):
    real = ousp.attention

    def strict(q, k, v, scale, causal=False, q_pos=None, k_pos=None, row_block=4096):
        if causal:  # the planted mistake: key j visible iff pos(j) < pos(i), diagonal excluded
            q_pos = (np.arange(q.shape[1]) if q_pos is None else np.asarray(q_pos)) - 1
        return real(q, k, v, scale, causal, q_pos, k_pos, row_block)

    monkeypatch.setattr(oracle, "attention", strict)
    assert _caught(ATTENTION_PINS)


# ------------------------------------------------------------------------------------------------
# planted mistakes in the ring merge
# ------------------------------------------------------------------------------------------------

def _pin_merge_logsumexp():
    # merging two partials of disjoint key sets gives the attention over their union
    D = 4
    q = RNG.standard_normal((1, 3, 1, D))
    k, v = RNG.standard_normal((1, 10, 1, D)), RNG.standard_normal((1, 10, 1, D))
    o1, l1 = oracle.attention(q, k[:, :4], v[:, :4], 0.5)
    o2, l2 = oracle.attention(q, k[:, 4:], v[:, 4:], 0.5)
    om, lm = oracle.merge(o1, l1, o2, l2)
    of, lf = oracle.attention(q, k, v, 0.5)
    assert np.allclose(om, of, atol=1e-13) and np.allclose(lm, lf, atol=1e-13)
    for i in range(3):  # lse of the union = log(exp(lse_1) + exp(lse_2))
        assert abs(math.log(math.exp(l1[0, i, 0]) + math.exp(l2[0, i, 0])) - lm[0, i, 0]) < 1e-12


def _pin_merge_empty():
    o = RNG.standard_normal((3, 4))
    l = RNG.standard_normal(3)
    om, lm = oracle.merge(o, l, np.zeros((3, 4)), np.full(3, NEG_INF))
    assert np.array_equal(om, o) and np.array_equal(lm, l)


MERGE_PINS = (_pin_merge_logsumexp, _pin_merge_empty)


def _merge_mutant(kind):
    def merge(prev_out, prev_lse, out, lse):
        prev_out, out = np.asarray(prev_out, float), np.asarray(out, float)
        prev_lse, lse = np.asarray(prev_lse, float), np.asarray(lse, float)
        d = np.where(np.isfinite(prev_lse) & np.isfinite(lse), lse - prev_lse, 0.0)
        if kind == "sigmoid argument sign":
            d_o = -d
        else:
            d_o = d
        res_out = prev_out - ousp._sigmoid(d_o)[..., None] * (prev_out - out)
        if kind == "logsigmoid sign":
            res_lse = prev_lse + ousp._logsigmoid(-d)
        elif kind == "lse not combined":
            res_lse = np.maximum(prev_lse, lse)
        else:
            res_lse = prev_lse - ousp._logsigmoid(-d)
        if kind != "empty partial not skipped":
            res_out = np.where(~np.isfinite(lse)[..., None], prev_out, res_out)
            res_lse = np.where(~np.isfinite(lse), prev_lse, res_lse)
        return res_out, res_lse
    return merge


MERGE_MUTANTS = ["sigmoid argument sign", "logsigmoid sign", "lse not combined",
                 "empty partial not skipped"]


def test_real_oracle_passes_every_merge_pin():
    assert _caught(MERGE_PINS) == []


@pytest.mark.parametrize("kind", MERGE_MUTANTS)
def test_merge_mutant_is_caught(kind, monkeypatch):
    monkeypatch.setattr(oracle, "merge", _merge_mutant(kind))
    assert _caught(MERGE_PINS), f"no pin catches: {kind}"


# ------------------------------------------------------------------------------------------------
# planted mistakes in the re-layout and the chunk orderings
# ------------------------------------------------------------------------------------------------

def _iota(B, S, H, D):
    b, t, h, d = np.meshgrid(np.arange(B), np.arange(S), np.arange(H), np.arange(D), indexing="ij")
    return ((b * 100000 + t) * 1000 + h) * 1000 + d


def _pack(x, lens):
    out, o = [], 0
    for n in lens:
        out.append(x[:, o:o + n].reshape(-1))
        o += n
    return np.concatenate(out)


def _pin_textbook_reshape():
    B, S, H, D, P = 2, 12, 6, 4, 3
    x = _iota(B, S, H, D)
    y = oracle.seq2head(_pack(x, [4, 4, 4]), B, H, D, [4, 4, 4])
    view = x.reshape(B, S, P, H // P, D)
    per = B * S * (H // P) * D
    for p in range(P):
        assert np.array_equal(y[p * per:(p + 1) * per].reshape(B, S, H // P, D), view[:, :, p])


def _pin_iota_uneven():
    B, H, D, lens, hc = 2, 5, 3, [5, 1, 7], [2, 2, 1]
    S = sum(lens)
    y = oracle.seq2head(_pack(_iota(B, S, H, D), lens), B, H, D, lens, hc)
    off, ho = 0, np.concatenate([[0], np.cumsum(hc)])
    for p in range(len(lens)):
        blk = y[off: off + B * S * hc[p] * D].reshape(B, S, hc[p], D)
        off += B * S * hc[p] * D
        bb, tt, hh, dd = np.meshgrid(np.arange(B), np.arange(S), np.arange(hc[p]), np.arange(D),
                                     indexing="ij")
        assert np.array_equal(blk, ((bb * 100000 + tt) * 1000 + hh + ho[p]) * 1000 + dd)


def _pin_round_trip():
    B, H, D, lens, hc = 3, 5, 2, [5, 1, 7], [2, 2, 1]
    src = np.random.default_rng(0).integers(0, 2**16, size=B * sum(lens) * H * D)
    back = oracle.head2seq(oracle.seq2head(src, B, H, D, lens, hc), B, H, D, lens, hc)
    assert np.array_equal(back, src)


def _pin_orders():
    zz = oracle.ring_positions("zigzag", 16, 4)
    assert zz[0].tolist() == [0, 1, 14, 15] and zz[3].tolist() == [6, 7, 8, 9]
    assert oracle.ring_positions("stripe", 20, 4)[1].tolist() == [1, 5, 9, 13, 17]
    for order in ("contiguous", "zigzag", "stripe"):
        pos = oracle.ring_positions(order, 17, 4)
        assert np.array_equal(np.sort(np.concatenate(pos)), np.arange(17))


LAYOUT_PINS = (_pin_textbook_reshape, _pin_iota_uneven, _pin_round_trip, _pin_orders)


def _caught_any(pins) -> list[str]:
    """Like _caught, but a crash (shape error, index error) also counts as caught."""
    failed = []
    for pin in pins:
        try:
            pin()
        except Exception:  # noqa: BLE001
            failed.append(pin.__name__)
    return failed


def _seq2head_mutant(kind):
    def seq2head(src, B, H, D, seq_lens, head_counts=None):
        P = len(seq_lens)
        head_counts = oracle.default_split(H, P) if head_counts is None else list(head_counts)
        so, ho = ousp._offsets(seq_lens), ousp._offsets(head_counts)
        S = so[-1]
        src = np.asarray(src).reshape(-1)
        dst = np.empty(B * S * H * D, dtype=src.dtype)
        chunks = [src[B * so[q] * H * D: B * so[q + 1] * H * D].reshape(B, seq_lens[q], H, D)
                  for q in range(P)]
        for p in range(P):
            base = B * S * ho[p] * D
            if kind == "head and sequence axes swapped":
                Y = dst[base: base + B * S * head_counts[p] * D].reshape(B, head_counts[p], S, D)
            else:
                Y = dst[base: base + B * S * head_counts[p] * D].reshape(B, S, head_counts[p], D)
            for q in range(P):
                g = ho[p] + (1 if kind == "head offset off by one" and p > 0 else 0)
                blk = chunks[q][:, :, g: g + head_counts[p], :]
                if kind == "head and sequence axes swapped":
                    Y[:, :, so[q]: so[q + 1], :] = blk.transpose(0, 2, 1, 3)
                elif kind == "sequence offset of the next rank":
                    o = so[(q + 1) % P]
                    Y[:, o: o + seq_lens[q], :, :] = blk
                else:
                    Y[:, so[q]: so[q + 1], :, :] = blk
        return dst
    return seq2head


LAYOUT_MUTANTS = ["head and sequence axes swapped", "head offset off by one",
                  "sequence offset of the next rank"]


def test_real_oracle_passes_every_layout_pin():
    assert _caught_any(LAYOUT_PINS) == []


@pytest.mark.parametrize("kind", LAYOUT_MUTANTS)
def test_layout_mutant_is_caught(kind, monkeypatch):
    monkeypatch.setattr(oracle, "seq2head", _seq2head_mutant(kind))
    assert _caught_any(LAYOUT_PINS), f"no pin catches: {kind}"


def test_zigzag_pairing_off_by_one_is_caught(monkeypatch):
    real = ousp.ring_positions

    def ring_positions(order, S, R):
        if order != "zigzag":
            return real(order, S, R)
        off = ousp._offsets(oracle.default_split(S, 2 * R))  # planted: piece 2R-2-r, not 2R-1-r
        return [np.concatenate([np.arange(off[r], off[r + 1]),
                                np.arange(off[(2 * R - 2 - r) % (2 * R)],
                                          off[(2 * R - 2 - r) % (2 * R) + 1])]) for r in range(R)]

    monkeypatch.setattr(oracle, "ring_positions", ring_positions)
    assert _caught_any(LAYOUT_PINS)


# ------------------------------------------------------------------------------------------------
# planted mistakes in the whole method (chunked + merged): caught by "equals unsplit attention"
# ------------------------------------------------------------------------------------------------

def _pin_chunked_equals_unsplit():
    # equal chunks (S = 24) first, so that a wrong mask shows as wrong values, then uneven ones
    for S, U, R, order, causal in ((24, 1, 3, "zigzag", True), (23, 1, 3, "zigzag", True),
                                   (23, 2, 2, "contiguous", True), (23, 1, 4, "stripe", False)):
        q, k, v = (RNG.standard_normal((1, S, 4, 4)) for _ in range(3))
        o, l = oracle.usp_attention(q, k, v, 0.5, causal, U, R, order)
        ro, rl = oracle.attention(q, k, v, 0.5, causal)
        assert np.allclose(o, ro, atol=1e-12) and np.allclose(l, rl, atol=1e-12)


def test_real_usp_attention_passes():
    assert _caught_any([_pin_chunked_equals_unsplit]) == []


def test_positions_swapped_in_a_ring_step_is_caught(monkeypatch):
    real = ousp.attention

    def swapped(q, k, v, scale, causal=False, q_pos=None, k_pos=None, row_block=4096):
        return real(q, k, v, scale, causal, k_pos if causal else q_pos,
                    q_pos if causal else k_pos, row_block)

    monkeypatch.setattr(ousp, "attention", swapped)
    try:  # on the equal-chunk case the swap runs and must give wrong values
        _pin_chunked_equals_unsplit()
        raise RuntimeError("not caught")
    except AssertionError:
        pass


def test_ring_partial_dropped_is_caught(monkeypatch):
    monkeypatch.setattr(ousp, "merge", lambda po, pl, o, l: (po, pl))  # keeps only the first step
    assert _caught_any([_pin_chunked_equals_unsplit])
