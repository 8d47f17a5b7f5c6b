"""Pins for the oracle's Ulysses re-layout and chunk orderings."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def iota(B, S, H, D):
    """Each element encodes its own (b, t, h, d)."""
    b, t, h, d = np.meshgrid(np.arange(B), np.arange(S), np.arange(H), np.arange(D), indexing="ij")
    return ((b * 100000 + t) * 1000 + h) * 1000 + d


def pack_chunks(x, lens):
    """Global [B][S][H][D] -> contiguous chunks back to back, each [B][s][H][D]."""
    out, o = [], 0
    for n in lens:
        out.append(x[:, o:o + n].reshape(-1))
        o += n
    return np.concatenate(out)


def test_even_split_equals_textbook_reshape():
    """Even split: head-sharded buffer p is the p-th head slice of the view [B][S][P][H/P][D]."""
    B, S, H, D, P = 2, 12, 6, 4, 3
    x = iota(B, S, H, D)
    y = oracle.seq2head(pack_chunks(x, [4, 4, 4]), B, H, D, [4, 4, 4])
    view = x.reshape(B, S, P, H // P, D)
    per = B * S * (H // P) * D
    for p in range(P):
        assert np.array_equal(y[p * per:(p + 1) * per].reshape(B, S, H // P, D), view[:, :, p])


@pytest.mark.parametrize("lens,heads", [([5, 1, 7], [2, 2, 1]), ([3, 3], None), ([1], None),
                                        ([0, 4, 2], [1, 3, 1]), ([6, 6, 6, 1], [2, 1, 1, 1])])
def test_iota_bijection(lens, heads):
    B, H, D = 2, 5, 3
    S = sum(lens)
    x = iota(B, S, H, D)
    P = len(lens)
    hc = heads or oracle.default_split(H, P)
    y = oracle.seq2head(pack_chunks(x, lens), B, H, D, lens, hc)
    # decode: every destination element must hold the source element with the same (b, t, h, d)
    off = 0
    ho = np.concatenate([[0], np.cumsum(hc)])
    for p in range(P):
        blk = y[off: off + B * S * hc[p] * D].reshape(B, S, hc[p], D)
        off += B * S * hc[p] * D
        bb, tt, hh, dd = np.meshgrid(np.arange(B), np.arange(S), np.arange(hc[p]), np.arange(D),
                                     indexing="ij")
        assert np.array_equal(blk, ((bb * 100000 + tt) * 1000 + hh + ho[p]) * 1000 + dd)
    assert sorted(y.tolist()) == sorted(x.reshape(-1).tolist())


@pytest.mark.parametrize("lens,heads", [([5, 1, 7], [2, 2, 1]), ([2, 9], None), ([4], None)])
def test_round_trip_identity(lens, heads):
    B, H, D = 3, 5, 2
    S = sum(lens)
    src = np.random.default_rng(0).integers(0, 2**16, size=B * S * H * D).astype(np.uint16)
    y = oracle.seq2head(src, B, H, D, lens, heads)
    back = oracle.head2seq(y, B, H, D, lens, heads)
    assert np.array_equal(back, src)
    assert np.array_equal(oracle.seq2head(back, B, H, D, lens, heads), y)


def test_p1_is_copy():
    x = np.arange(2 * 7 * 3 * 4)
    assert np.array_equal(oracle.seq2head(x, 2, 3, 4, [7]), x)
    assert np.array_equal(oracle.head2seq(x, 2, 3, 4, [7]), x)


def test_golden_splits():
    g = json.load(open(os.path.join(GOLDEN, "workload_splits.json")))
    for case in g["splits"]:
        assert oracle.default_split(case["S"], case["P"]) == case["lens"]
    for key in ("flux_1008_tokens", "flux_1024_tokens", "qwen_1328_tokens"):
        c = g[key]
        assert c["image_side_latent"] ** 2 == c["image"] and c["text"] + c["image"] == c["total"]


@pytest.mark.parametrize("order", ["contiguous", "zigzag", "stripe"])
@pytest.mark.parametrize("S,R", [(1, 1), (10, 3), (64, 8), (17, 4), (5, 8)])
def test_orders_are_bijections_and_increasing(order, S, R):
    pos = oracle.ring_positions(order, S, R)
    allp = np.concatenate(pos)
    assert np.array_equal(np.sort(allp), np.arange(S))
    for p in pos:
        assert np.all(np.diff(p) > 0)


def test_order_closed_forms():
    S, R = 20, 4
    assert all(np.array_equal(a, b) for a, b in
               zip(oracle.ring_positions("zigzag", S, 1), oracle.ring_positions("contiguous", S, 1)))
    zz = oracle.ring_positions("zigzag", 16, 4)   # pieces of 2: rank r holds pieces r and 7-r
    assert zz[0].tolist() == [0, 1, 14, 15] and zz[3].tolist() == [6, 7, 8, 9]
    st = oracle.ring_positions("stripe", S, R)
    assert st[1].tolist() == [1, 5, 9, 13, 17]
    big = oracle.ring_positions("zigzag", 65536, 8)
    assert all(len(p) == 8192 for p in big)
    assert big[0][4095] == 4095 and big[0][4096] == 15 * 4096


def test_virtual_rank_lengths():
    assert oracle.virtual_rank_lengths("contiguous", 7145, 2, 2) == [1787, 1786, 1786, 1786]
    with pytest.raises(ValueError):
        oracle.virtual_rank_lengths("contiguous", 10, 2, 1, [3, 3])
