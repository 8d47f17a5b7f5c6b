"""usp_attention end to end (re-layout, partial attention, merge, inverse re-layout) against the
fp64 oracle, on small grids element by element and on the full-size workloads by sampled heads
and rows."""
import math

import numpy as np
import pytest

import oracle
from sequence_attention_tcgen05_gb300 import synth, usp

from gpu_util import check_attention, to_dev_bf16, torch, widen

pytestmark = pytest.mark.gpu


def run_usp(B, S, H, D, U, R, causal=False, order="contiguous", seq_lens=None, head_counts=None,
            seed=0, text_rows=0, text_scale=1.0, out="fp32"):
    t = torch()
    qb, kb, vb = synth.make_qkv_bits(B, S, H, D, seed, text_rows, text_scale)
    q, k, v = to_dev_bf16(qb), to_dev_bf16(kb), to_dev_bf16(vb)
    dt = t.float32 if out == "fp32" else t.bfloat16
    o, lse = usp.attention(q, k, v, causal=causal, ulysses_degree=U, ring_degree=R, order=order,
                           seq_lens=seq_lens, head_counts=head_counts, out_dtype=dt)
    t.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy(), (qb, kb, vb)


def test_tiny_ring3_config():
    """B=1, H=4, D=64, S=1000 over 3 ring ranks (334/333/333), non-causal, fp32 O and LSE."""
    o, l, (qb, kb, vb) = run_usp(1, 1000, 4, 64, 1, 3, seq_lens=[334, 333, 333])
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / 8)
    check_attention(o, l, ro, rl, "tiny ring 3")


def test_tiny_uaa3_config():
    """Same tensors as Ulysses Anything over 3 ranks: heads 2/1/1, lengths 334/333/333."""
    o, l, (qb, kb, vb) = run_usp(1, 1000, 4, 64, 3, 1, seq_lens=[334, 333, 333],
                                 head_counts=[2, 1, 1])
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / 8)
    check_attention(o, l, ro, rl, "tiny uaa 3")


GRID = []
for (U, R) in [(1, 1), (2, 1), (3, 1), (1, 2), (1, 3), (2, 2), (2, 3), (1, 8), (4, 4)]:
    for order in ["contiguous", "zigzag", "stripe"]:
        GRID.append((U, R, order))


@pytest.mark.parametrize("U,R,order", GRID)
@pytest.mark.parametrize("causal", [False, True])
def test_grid_small(U, R, order, causal):
    B, S, H, D = (2, 523, 5, 64) if (U + R) % 2 else (1, 777, 4, 128)
    if H < U:
        H = U
    o, l, (qb, kb, vb) = run_usp(B, S, H, D, U, R, causal, order, seed=U * 10 + R)
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / math.sqrt(D), causal)
    check_attention(o, l, ro, rl, f"grid U={U} R={R} {order} causal={causal}")


@pytest.mark.parametrize("B,S,H,D,U,R,causal", [
    (1, 512, 4, 64, 1, 2, True),      # half-chunks of 128 rows: one tile each
    (2, 2048, 4, 128, 2, 4, True),    # half-chunks of 256 rows, Ulysses 2 x ring 4
    (1, 3072, 3, 128, 1, 3, True),    # half-chunks of 512 rows, ring 3
    (2, 1024, 4, 64, 2, 2, False),    # non-causal zigzag
])
def test_zigzag_in_place_half_chunks(B, S, H, D, U, R, causal):
    """Zigzag ring chunks of two equal half-chunks of whole 128-row tiles are read in place by
    two-piece tensor maps (no workspace copy); checked element by element against the oracle."""
    assert S % (2 * R) == 0 and (S // (2 * R)) % 128 == 0
    o, l, (qb, kb, vb) = run_usp(B, S, H, D, U, R, causal, "zigzag", seed=S + R)
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / math.sqrt(D), causal)
    check_attention(o, l, ro, rl, f"zigzag in place S={S} U={U} R={R} causal={causal}")
    ws = usp.usp_attention_workspace_size(B, S, H, D, U, R, "zigzag", usp.USP_FP32)
    # status word + ring partials only: no Q/K/V copies
    rows_h = B * S * H
    assert ws < 256 + R * (rows_h * D * 4 + rows_h * 4) + 4096 * R + 2 ** 20


def test_uneven_seq_lens_and_bf16_out():
    S, U, R = 1001, 2, 2
    ring = oracle.default_split(S, R)
    lens = [1, ring[0] - 1, ring[1] - 300, 300]
    o, l, (qb, kb, vb) = run_usp(1, S, 6, 128, U, R, True, seq_lens=lens, head_counts=[5, 1],
                                 out="bf16")
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / math.sqrt(128), True)
    check_attention(o, l, ro, rl, "uneven + bf16")


def _check_heads(w: synth.Workload, heads, rows=None):
    o, l, (qb, kb, vb) = run_usp(w.B, w.S, w.H, w.D, w.ulysses_degree, w.ring_degree, w.causal,
                                 w.order, list(w.seq_lens) or None, seed=w.seed,
                                 text_rows=w.text_rows, text_scale=w.text_scale)
    scale = 1 / math.sqrt(w.D)
    for h in heads:
        k = widen(kb[0, :, h]); v = widen(vb[0, :, h])
        idx = np.arange(w.S) if rows is None else rows
        ro, rl = oracle.attention_rows(widen(qb[0, idx, h]), k, v, scale, w.causal, idx)
        check_attention(o[0, idx, h], l[0, idx, h], ro, rl, f"{w.name} head {h}")


@pytest.mark.parametrize("name,heads", [("flux_1024_u2", [0, 11, 12, 23]),
                                        ("flux_1008_uaa2", [0, 12, 23]),
                                        ("flux_1008_uaa3", [0, 8, 16, 23]),
                                        ("qwen_1328_u2r2", [0, 12, 23])])
def test_full_size_workloads(name, heads):
    _check_heads(synth.WORKLOADS[name], heads)


def test_long_context_causal_zigzag_sampled():
    w = synth.WORKLOADS["llm_64k_ring8_zigzag"]
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.integers(0, w.S, 512), np.arange(0, 130),
                                     np.arange(w.S - 130, w.S), 4096 * np.arange(1, 16) - 1,
                                     4096 * np.arange(1, 16)]))
    _check_heads(w, [0, 31], rows)
