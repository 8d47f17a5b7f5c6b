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
        for mode in (["fused", "separate"] if R > 1 else ["none"]):
            GRID.append((U, R, order, mode))


def set_ring_mode(monkeypatch, mode):
    """Pins how usp_attention runs the ring steps (the library otherwise picks by its time
    model): "fused" = one online softmax per query block across all ring steps, "separate" =
    per-step fp32 partials and a merge pass."""
    if mode in ("fused", "separate"):
        monkeypatch.setenv("USP_RING_MERGE", mode)


@pytest.mark.parametrize("U,R,order,mode", GRID)
@pytest.mark.parametrize("causal", [False, True])
def test_grid_small(U, R, order, mode, causal, monkeypatch):
    set_ring_mode(monkeypatch, mode)
    B, S, H, D = (2, 523, 5, 64) if (U + R) % 2 else (1, 777, 4, 128)
    if H < U:
        H = U
    o, l, (qb, kb, vb) = run_usp(B, S, H, D, U, R, causal, order, seed=U * 10 + R)
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / math.sqrt(D), causal)
    check_attention(o, l, ro, rl, f"grid U={U} R={R} {order} causal={causal} ring={mode}")


@pytest.mark.parametrize("B,U,R,order,S,k", [
    (1, 1, 2, "contiguous", 1000, 1), (1, 2, 2, "contiguous", 1537, 2), (1, 1, 3, "stripe", 777, 1),
    (1, 2, 2, "zigzag", 1000, 1), (1, 1, 4, "zigzag", 1537, 9), (1, 3, 2, "contiguous", 2000, 3),
    (2, 2, 2, "contiguous", 1100, 2), (2, 1, 3, "zigzag", 900, 1),
])
@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_split_fused_ring(B, U, R, order, S, k, out, monkeypatch):
    """A fused non-causal ring with the last k 256-row blocks of its last ring chunk (last Ulysses
    group) run as separate ring steps: their fp32 partials are merged after the attention, while
    every other query block carries its chain (k = 9 splits the whole chunk; B = 2 checks the
    batch stride of the split rows' slots)."""
    monkeypatch.setenv("USP_RING_MERGE", "fused")
    monkeypatch.setenv("USP_RING_SPLIT", str(k))
    H, D = max(2 * U, 4), 128
    ws = usp.usp_attention_workspace_size(B, S, H, D, U, R, order, usp.USP_FP32, False)
    assert ws > 256  # the split rows' partial slots
    o, l, (qb, kb, vb) = run_usp(B, S, H, D, U, R, False, order, seed=S + k, out=out)
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / math.sqrt(D), False)
    check_attention(o, l, ro, rl, f"split fused ring U={U} R={R} {order} S={S} k={k} {out}")


@pytest.mark.parametrize("mode", ["fused", "separate"])
@pytest.mark.parametrize("B,S,H,D,U,R,causal", [
    (1, 512, 4, 64, 1, 2, True),      # half-chunks of 128 rows: one tile each
    (2, 2048, 4, 128, 2, 4, True),    # half-chunks of 256 rows, Ulysses 2 x ring 4
    (1, 3072, 3, 128, 1, 3, True),    # half-chunks of 512 rows, ring 3
    (1, 1536, 2, 128, 1, 2, True),    # half-chunks of 384 rows: a 256-row block spans both
    (2, 1024, 4, 64, 2, 2, False),    # non-causal zigzag
])
def test_zigzag_in_place_half_chunks(B, S, H, D, U, R, causal, mode, monkeypatch):
    """Zigzag ring chunks of two equal half-chunks of whole 128-row tiles are read in place by
    two-piece tensor maps (no workspace copy); checked element by element against the oracle."""
    set_ring_mode(monkeypatch, mode)
    assert S % (2 * R) == 0 and (S // (2 * R)) % 128 == 0
    o, l, (qb, kb, vb) = run_usp(B, S, H, D, U, R, causal, "zigzag", seed=S + R)
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / math.sqrt(D), causal)
    check_attention(o, l, ro, rl, f"zigzag in place S={S} U={U} R={R} causal={causal} ring={mode}")
    ws = usp.usp_attention_workspace_size(B, S, H, D, U, R, "zigzag", usp.USP_FP32, causal)
    # status word (+ ring partials when separate) only: no Q/K/V copies
    rows_h = B * S * H
    if mode == "fused":
        assert ws == 256
    else:
        assert ws < 256 + R * (rows_h * D * 4 + rows_h * 4) + 4096 * R + 2 ** 20


@pytest.mark.parametrize("mode", ["fused", "separate"])
def test_uneven_seq_lens_and_bf16_out(mode, monkeypatch):
    set_ring_mode(monkeypatch, mode)
    S, U, R = 1001, 2, 2
    ring = oracle.default_split(S, R)
    lens = [1, ring[0] - 1, ring[1] - 300, 300]
    o, l, (qb, kb, vb) = run_usp(1, S, 6, 128, U, R, True, seq_lens=lens, head_counts=[5, 1],
                                 out="bf16")
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / math.sqrt(128), True)
    check_attention(o, l, ro, rl, "uneven + bf16")


_INPUTS = {}


def _workload_inputs(w: synth.Workload):
    """The workload's seeded Q, K, V bits, generated once per test module (the 64K inputs take a
    while to generate on the host)."""
    key = (w.B, w.S, w.H, w.D, w.seed, w.text_rows, w.text_scale)
    if key not in _INPUTS:
        _INPUTS.clear()
        _INPUTS[key] = synth.make_qkv_bits(w.B, w.S, w.H, w.D, w.seed, w.text_rows, w.text_scale)
    return _INPUTS[key]


def _check_heads(w: synth.Workload, heads, rows=None):
    t = torch()
    qb, kb, vb = _workload_inputs(w)
    q, k, v = to_dev_bf16(qb), to_dev_bf16(kb), to_dev_bf16(vb)
    o, l = usp.attention(q, k, v, causal=w.causal, ulysses_degree=w.ulysses_degree,
                         ring_degree=w.ring_degree, order=w.order,
                         seq_lens=list(w.seq_lens) or None, out_dtype=t.float32)
    t.cuda.synchronize()
    o, l = o.cpu().numpy(), l.cpu().numpy()
    del q, k, v
    scale = 1 / math.sqrt(w.D)
    for h in heads:
        k = widen(kb[0, :, h]); v = widen(vb[0, :, h])
        idx = np.arange(w.S) if rows is None else rows
        ro, rl = oracle.attention_rows(widen(qb[0, idx, h]), k, v, scale, w.causal, idx)
        check_attention(o[0, idx, h], l[0, idx, h], ro, rl, f"{w.name} head {h}")


@pytest.mark.parametrize("name,heads", [("flux_1024_u2", [0, 11, 12, 23]),
                                        ("flux_1008_uaa2", [0, 12, 23]),
                                        ("flux_1008_uaa3", [0, 8, 16, 23])])
def test_full_size_workloads(name, heads):
    _check_heads(synth.WORKLOADS[name], heads)


@pytest.mark.parametrize("mode", ["fused", "separate"])
def test_full_size_qwen(mode, monkeypatch):
    set_ring_mode(monkeypatch, mode)
    _check_heads(synth.WORKLOADS["qwen_1328_u2r2"], [0, 12, 23])


@pytest.mark.parametrize("mode", ["fused", "separate"])
def test_long_context_causal_zigzag_sampled(mode, monkeypatch):
    set_ring_mode(monkeypatch, mode)
    w = synth.WORKLOADS["llm_64k_ring8_zigzag"]
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.integers(0, w.S, 512), np.arange(0, 130),
                                     np.arange(w.S - 130, w.S), 4096 * np.arange(1, 16) - 1,
                                     4096 * np.arange(1, 16)]))
    _check_heads(w, [0, 31], rows)


def _sampled_rows(w, n=512, seed=0):
    """Random rows plus the first and last rows and both sides of every ring chunk boundary."""
    rng = np.random.default_rng(seed)
    bounds = set()
    for pos in oracle.ring_positions(w.order, w.S, w.ring_degree):
        steps = np.flatnonzero(np.diff(pos) != np.diff(pos)[:1]) if len(pos) > 1 else []
        for i in [0, len(pos) - 1, *steps, *(np.asarray(steps) + 1)]:
            if 0 <= i < len(pos):
                bounds.add(int(pos[i]))
    return np.unique(np.concatenate([rng.integers(0, w.S, n), np.arange(0, 130),
                                     np.arange(w.S - 130, w.S), np.array(sorted(bounds))]))


@pytest.mark.parametrize("mode", ["fused", "separate"])
@pytest.mark.parametrize("name", ["llm_64k257_ring8_zigzag", "llm_32k_ring4_stripe"])
def test_anything_large_uneven_causal(name, mode, monkeypatch):
    """Ring Anything at large, uneven causal sizes: 65793 tokens over a zigzag ring of 8 (half-
    chunks of 4111/4112 rows, read through span maps) and 32771 tokens over a stripe ring of 4;
    sampled rows (every half-chunk boundary among them) of two heads against the oracle."""
    set_ring_mode(monkeypatch, mode)
    w = synth.WORKLOADS[name]
    _check_heads(w, [0, w.H - 1], _sampled_rows(w))


def test_ulysses_anything_24_heads_over_5():
    """24 heads over 5 Ulysses ranks (5/5/5/5/4) at FLUX 1024^2 length: every head of the last,
    smaller group and the heads on both sides of each group boundary, all rows."""
    w = synth.WORKLOADS["flux_1024_uaa5"]
    _check_heads(w, [0, 4, 5, 9, 10, 14, 15, 19, 20, 21, 22, 23])


@pytest.mark.parametrize("U,R,order,causal,mode", [
    (1, 1, "contiguous", False, "none"), (2, 1, "contiguous", True, "none"),
    (1, 3, "zigzag", True, "fused"), (1, 3, "zigzag", True, "separate"),   # ragged: span maps
    (2, 2, "stripe", True, "fused"), (1, 2, "zigzag", True, "separate"),
    (3, 2, "contiguous", False, "fused"),
])
def test_qkvpacked_matches_oracle(U, R, order, causal, mode, monkeypatch):
    """usp_attention_qkvpacked on a [B][S][3][H][D] input: the tensor maps read the packed rows in
    place (3*H*D row stride), for zigzag chunks of whole-tile and of ragged half-chunks alike."""
    set_ring_mode(monkeypatch, mode)
    t = torch()
    B, S, H, D = (2, 1000, 4, 128) if order != "zigzag" or R != 2 else (1, 1024, 3, 128)
    qb, kb, vb = synth.make_qkv_bits(B, S, H, D, seed=7)
    packed = np.ascontiguousarray(np.stack([qb, kb, vb], axis=2))  # [B][S][3][H][D]
    qkv = to_dev_bf16(packed)
    o = t.empty((B, S, H, D), dtype=t.float32, device="cuda")
    lse = t.empty((B, S, H), dtype=t.float32, device="cuda")
    nbytes = usp.usp_attention_workspace_size(B, S, H, D, U, R, order, usp.USP_FP32, causal)
    ws = t.zeros(nbytes, dtype=t.uint8, device="cuda")
    usp.usp_attention_qkvpacked(qkv, B, S, H, D, 1 / math.sqrt(D), causal, U, R, o, lse, ws,
                                nbytes, order=order)
    assert usp.usp_check_status(ws) == usp.USP_OK
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / math.sqrt(D), causal)
    check_attention(o.cpu().numpy(), lse.cpu().numpy(), ro, rl,
                    f"qkvpacked U={U} R={R} {order} causal={causal} ring={mode}")


@pytest.mark.parametrize("mode", ["fused", "separate"])
@pytest.mark.parametrize("S,H,U,R,order,causal", [
    (1, 2, 1, 8, "zigzag", True),       # one token, seven empty ring chunks
    (5, 2, 1, 8, "zigzag", True),       # fewer tokens than half-chunks
    (7, 3, 1, 16, "stripe", True),      # fewer tokens than ring ranks
    (130, 4, 4, 4, "contiguous", True),  # 16 virtual ranks, one head each
    (129, 4, 4, 4, "zigzag", False),
    (2, 1, 1, 2, "contiguous", False),  # one query per rank
])
def test_degenerate_shapes(S, H, U, R, order, causal, mode, monkeypatch):
    set_ring_mode(monkeypatch, mode)
    o, l, (qb, kb, vb) = run_usp(1, S, H, 128, U, R, causal, order, seed=S)
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / math.sqrt(128), causal)
    check_attention(o, l, ro, rl, f"degenerate S={S} U={U} R={R} {order} causal={causal} ring={mode}")


def test_largest_ring_256k_causal_zigzag():
    """The largest ring the library runs (16 ranks) on a 256K-token causal sequence (8 heads of
    128; 32 half-chunks of 8192 rows, addressed in place), fused ring steps: sampled rows of the
    first and last heads against the oracle."""
    w = synth.Workload("llm_256k_ring16_zigzag", 1, 8, 128, 262144, 1, 16, causal=True,
                       order="zigzag")
    assert usp.usp_attention_ring_mode(w.B, w.S, w.H, w.D, True, 1, 16, "zigzag",
                                       usp.USP_FP32) == "fused"
    rows = _sampled_rows(w, n=256)
    _check_heads(w, [0, w.H - 1], rows)


def test_repeated_calls_on_the_same_buffers(monkeypatch):
    """A call that repeats the previous one (same shapes, buffers and settings) relaunches the
    kernel parameters built then: new input contents in the same buffers must still give the right
    result, and a changed ring-mode override must not reuse them."""
    t = torch()
    B, S, H, D, U, R = 1, 1537, 4, 128, 2, 3
    scale = 1 / math.sqrt(D)
    q, k, v = (t.empty((B, S, H, D), dtype=t.bfloat16, device="cuda") for _ in range(3))
    o = t.empty((B, S, H, D), dtype=t.float32, device="cuda")
    lse = t.empty((B, S, H), dtype=t.float32, device="cuda")
    monkeypatch.setenv("USP_RING_MERGE", "separate")  # the larger workspace of the two modes
    nbytes = usp.usp_attention_workspace_size(B, S, H, D, U, R, "zigzag", usp.USP_FP32, True)
    ws = t.zeros(nbytes, dtype=t.uint8, device="cuda")
    for seed, mode in ((1, "separate"), (2, "separate"), (3, "fused"), (4, "fused")):
        monkeypatch.setenv("USP_RING_MERGE", mode)
        qb, kb, vb = synth.make_qkv_bits(B, S, H, D, seed)
        for dst, bits in zip((q, k, v), (qb, kb, vb)):
            dst.copy_(to_dev_bf16(bits))
        usp.usp_attention(q, k, v, B, S, H, D, scale, True, U, R, o, lse, ws, nbytes, order="zigzag")
        assert usp.usp_check_status(ws) == usp.USP_OK
        ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), scale, True)
        check_attention(o.cpu().numpy(), lse.cpu().numpy(), ro, rl, f"repeat seed={seed} ring={mode}")


@pytest.mark.parametrize("B,S,H,D,U,R,causal,order,split,deal", [
    (2, 1570, 4, 64, 1, 3, True, "zigzag", None, 1),       # round-robin beats the snake
    (2, 2152, 2, 64, 1, 4, True, "zigzag", None, 2),       # odd heads visit their blocks in reverse
    (2, 1085, 3, 64, 1, 4, True, "contiguous", None, 3),   # both
    (2, 600, 3, 64, 1, 4, True, "zigzag", None, 4),        # dynamic: the CTA free first
    (1, 3000, 16, 64, 1, 4, True, "stripe", None, 4),
    (1, 2600, 16, 128, 2, 2, False, "contiguous", 2, 0),   # split fused ring: a second unit group
])
@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_unit_deals_bit_identical(B, S, H, D, U, R, causal, order, split, deal, out, monkeypatch):
    """The deal (which CTA takes which work unit, and in which order each head visits its query
    blocks) changes only the timing: every forced deal gives the bits of the library's own
    choice, which is the one its time model names and matches the oracle.  Every case has more
    units than a GB300 has SMs, so the deals differ from the second round on."""
    monkeypatch.delenv("USP_UNIT_DEAL", raising=False)
    if split is not None:
        monkeypatch.setenv("USP_RING_SPLIT", str(split))
    o_dt = usp.USP_FP32 if out == "fp32" else usp.USP_BF16
    chosen = usp.usp_plan_deals(B, S, H, D, causal, U, R, order, o_dt)
    assert [d for _, d, _, _ in chosen] == [deal] and chosen[0][0] > 152
    o, l, (qb, kb, vb) = run_usp(B, S, H, D, U, R, causal, order, seed=31, out=out)
    for forced in range(8):
        monkeypatch.setenv("USP_UNIT_DEAL", str(forced))
        assert [d for _, d, _, _ in usp.usp_plan_deals(B, S, H, D, causal, U, R, order, o_dt)] == \
            [forced] * len(chosen)
        o2, l2, _ = run_usp(B, S, H, D, U, R, causal, order, seed=31, out=out)
        assert np.array_equal(o2.view(np.uint32), o.view(np.uint32)), forced
        assert np.array_equal(l2.view(np.uint32), l.view(np.uint32)), forced
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), 1 / math.sqrt(D), causal)
    check_attention(o, l, ro, rl, f"deal {chosen} {order} causal={causal} out={out}")


def test_dynamic_deal_counter(monkeypatch):
    """The dynamic deal's counter (workspace bytes 8-15): four calls back to back on the same
    buffers and workspace, with no host synchronisation between them (fresh inputs copied in
    and each output copied out in the stream), each start from zero, left there by the launch
    before (every output matches the oracle); a launch whose waits run out
    (USP_TEST_WITHHOLD_LOADS: no unit is ever handed out) still leaves it at zero, and the next
    call on the same workspace is correct."""
    t = torch()
    B, S, H, D, U, R = 2, 600, 3, 64, 1, 4
    scale = 1 / math.sqrt(D)
    monkeypatch.setenv("USP_UNIT_DEAL", "4")
    assert [d for _, d, _, _ in usp.usp_plan_deals(B, S, H, D, True, U, R, "zigzag", usp.USP_FP32)] == [4]
    nbytes = usp.usp_attention_workspace_size(B, S, H, D, U, R, "zigzag", usp.USP_FP32, True)
    ws = t.zeros(nbytes, dtype=t.uint8, device="cuda")
    ws[8:16] = 0x5A  # not zero: the first call with this workspace clears it in the stream
    bits = [synth.make_qkv_bits(B, S, H, D, 40 + seed) for seed in range(4)]
    dev = [tuple(to_dev_bf16(x) for x in b) for b in bits]
    q, k, v = (t.empty_like(x) for x in dev[0])
    o = t.empty((B, S, H, D), dtype=t.float32, device="cuda")
    lse = t.empty((B, S, H), dtype=t.float32, device="cuda")
    saved = []
    t.cuda.synchronize()
    for dq, dk, dv in dev:
        q.copy_(dq)
        k.copy_(dk)
        v.copy_(dv)
        usp.usp_attention(q, k, v, B, S, H, D, scale, True, U, R, o, lse, ws, nbytes, order="zigzag")
        saved.append((o.clone(), lse.clone()))
    assert usp.usp_check_status(ws) == usp.USP_OK
    assert int(ws[8:16].view(t.int32).abs().sum()) == 0
    for (qb, kb, vb), (so, sl) in zip(bits, saved):
        ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), scale, True)
        check_attention(so.cpu().numpy(), sl.cpu().numpy(), ro, rl, "dynamic deal, back to back")
    monkeypatch.setenv("USP_WAIT_BUDGET_MS", "50")
    monkeypatch.setenv("USP_TEST_WITHHOLD_LOADS", "1")
    usp.usp_attention(q, k, v, B, S, H, D, scale, True, U, R, o, lse, ws, nbytes, order="zigzag")
    assert usp.usp_check_status(ws) == usp.USP_ERR_TIMEOUT
    assert int(ws[8:16].view(t.int32).abs().sum()) == 0
    monkeypatch.delenv("USP_TEST_WITHHOLD_LOADS")
    monkeypatch.delenv("USP_WAIT_BUDGET_MS")
    o.fill_(0)
    usp.usp_attention(q, k, v, B, S, H, D, scale, True, U, R, o, lse, ws, nbytes, order="zigzag")
    assert usp.usp_check_status(ws) == usp.USP_OK
    qb, kb, vb = bits[-1]
    ro, rl = oracle.attention(widen(qb), widen(kb), widen(vb), scale, True)
    check_attention(o.cpu().numpy(), lse.cpu().numpy(), ro, rl, "dynamic deal after a timed-out launch")
