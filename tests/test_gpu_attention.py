"""usp_attn_partial (tcgen05 kernel) against the fp64 oracle on the same seeded bf16 inputs."""
import math
import time

import numpy as np
import pytest

import oracle
from sequence_attention_tcgen05_gb300 import synth, usp

from gpu_util import Guarded, check_attention, to_dev_bf16, torch, widen

pytestmark = pytest.mark.gpu


def run_partial(B, H, Sq, Sk, D, q_pos=None, k_pos=None, seed=0, out="fp32", packed=False,
                k_row_scale=None):
    t = torch()
    qb = synth.make_tensor_bits(seed, 0, B, Sq, H, D)
    kb = synth.make_tensor_bits(seed, 1, B, Sk, H, D)
    vb = synth.make_tensor_bits(seed, 2, B, Sk, H, D)
    if k_row_scale is not None:  # key row t multiplied by k_row_scale[t] in fp32, then bf16 again
        kb = synth.bf16_bits(synth.bf16_to_f32(kb) * np.float32(k_row_scale)[None, :, None, None])
    if packed:
        # q, k, v rows interleaved as [B][S][3][H][D] (QKV-packed layout): row stride 3*H*D
        assert Sq == Sk
        pk = np.stack([qb, kb, vb], axis=2)
        dev = to_dev_bf16(pk.reshape(-1))
        n3 = H * D
        q, k, v = dev[0:], dev[n3:], dev[2 * n3:]
        qs = ks = 3 * H * D
    else:
        q, k, v = to_dev_bf16(qb), to_dev_bf16(kb), to_dev_bf16(vb)
        qs = ks = H * D
    dt = t.float32 if out == "fp32" else t.bfloat16
    o = Guarded((B, Sq, H, D), dt)
    lse = Guarded((B, Sq, H), t.float32)
    status = t.zeros(1, dtype=t.int32, device="cuda")
    scale = 1.0 / math.sqrt(D)
    qp = usp.Positions.make(*q_pos) if q_pos else None
    kp = usp.Positions.make(*k_pos) if k_pos else None
    usp.usp_attn_partial(q, k, v, B, H, Sq, Sk, D, qs, ks, scale, o.view, lse.view, qp, kp,
                         status=status)
    assert usp.usp_check_status(status) == usp.USP_OK
    o.check()
    lse.check()
    return (o.view.float().cpu().numpy(), lse.view.cpu().numpy(),
            widen(qb), widen(kb), widen(vb), scale)


def positions(spec):
    segs, stride = spec
    return np.concatenate([s + stride * np.arange(n) for s, n in segs]).astype(np.int64)


@pytest.mark.parametrize("B,H,Sq,Sk,D", [
    (1, 1, 128, 128, 128), (1, 1, 128, 128, 64), (1, 2, 200, 333, 64), (2, 3, 257, 129, 128),
    (1, 1, 1, 1, 64), (1, 2, 5, 700, 128), (1, 4, 1000, 1000, 64), (1, 2, 384, 2500, 128)])
def test_noncausal(B, H, Sq, Sk, D):
    o, l, q, k, v, scale = run_partial(B, H, Sq, Sk, D)
    ro, rl = oracle.attention(q, k, v, scale)
    check_attention(o, l, ro, rl, f"noncausal {B},{H},{Sq},{Sk},{D}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("qspec,kspec", [
    (([(0, 300)], 1), ([(0, 300)], 1)),                       # diagonal chunk
    (([(500, 260)], 1), ([(0, 700)], 1)),                     # later q chunk, mixed tiles
    (([(0, 130)], 1), ([(200, 150)], 1)),                     # q entirely before k: all masked
    (([(0, 100), (700, 100)], 1), ([(0, 100), (700, 100)], 1)),   # zigzag, own rank
    (([(0, 100), (700, 100)], 1), ([(100, 100), (600, 100)], 1)),  # zigzag, other rank
    (([(1, 150)], 4), ([(3, 150)], 4)),                       # stripe, r < r2
    (([(3, 150)], 4), ([(1, 150)], 4)),                       # stripe, r > r2
])
def test_causal_positions(D, qspec, kspec):
    Sq = sum(n for _, n in qspec[0])
    Sk = sum(n for _, n in kspec[0])
    o, l, q, k, v, scale = run_partial(1, 2, Sq, Sk, D, qspec, kspec, seed=5)
    ro, rl = oracle.attention(q, k, v, scale, True, positions(qspec), positions(kspec))
    check_attention(o, l, ro, rl, f"causal {qspec} {kspec}")


def test_empty_kv_chunk():
    t = torch()
    B, H, Sq, D = 1, 2, 150, 64
    qb = synth.make_tensor_bits(0, 0, B, Sq, H, D)
    q = to_dev_bf16(qb)
    kv = to_dev_bf16(qb[:, :1])
    o = Guarded((B, Sq, H, D), t.float32)
    lse = Guarded((B, Sq, H), t.float32)
    usp.usp_attn_partial(q, kv, kv, B, H, Sq, 0, D, H * D, H * D, 0.125, o.view, lse.view)
    t.cuda.synchronize()
    o.check()
    assert bool((o.view == 0).all()) and bool(t.isneginf(lse.view).all())


def test_bf16_output_and_packed_qkv():
    o, l, q, k, v, scale = run_partial(2, 3, 300, 300, 128, out="bf16", packed=True)
    ro, rl = oracle.attention(q, k, v, scale)
    check_attention(o, l, ro, rl, "bf16 packed")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B,H,Sq,Sk,causal", [
    (1, 1, 1, 1, False), (2, 3, 131, 200, False), (1, 2, 300, 129, False), (1, 5, 517, 700, False),
    (2, 2, 300, 300, True), (1, 3, 133, 133, True)])
def test_bf16_output_every_element(B, H, Sq, Sk, D, causal):
    """bf16 O is written as 16-byte stores after a word transpose across the four threads of each
    row: every element of every valid row must be written (an element left at the canary fill
    fails the comparison) and nothing around the buffer touched, for ragged row counts."""
    spec = (([(0, Sq)], 1), ([(0, Sk)], 1)) if causal else (None, None)
    o, l, q, k, v, scale = run_partial(B, H, Sq, Sk, D, spec[0], spec[1], seed=11, out="bf16")
    if causal:
        ro, rl = oracle.attention(q, k, v, scale, True, positions(spec[0]), positions(spec[1]))
    else:
        ro, rl = oracle.attention(q, k, v, scale)
    check_attention(o, l, ro, rl, f"bf16 out {B},{H},{Sq},{Sk},{D} causal={causal}")


def test_repeat_calls_identical():
    a = run_partial(1, 4, 640, 900, 128, seed=9)
    b = run_partial(1, 4, 640, 900, 128, seed=9)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def key_profile(kind, Sk):
    t = np.arange(Sk, dtype=np.float64)
    if kind == "rising":    # key norms grow 16x along the keys: the row max climbs tile after tile
        return 2.0 ** (4.0 * t / Sk)
    if kind == "falling":   # the first tiles dominate: later exponentials are tiny against m
        return 2.0 ** (4.0 * (1.0 - t / Sk))
    f = np.ones(Sk)         # a few large keys late in the row
    f[[260, 261, 500, 777, 901, Sk - 10]] = 20.0
    return f


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind", ["rising", "falling", "spikes"])
@pytest.mark.parametrize("causal", [False, True])
def test_running_max_changes(D, kind, causal):
    """Scores that rise far above the first key tile's maximum force the softmax's slow path
    (running max raised, O rescaled in TMEM, exponentials redone); falling scores keep a stale
    maximum far above later tiles.  Both are exact after the final division by the row sum."""
    Sq, Sk = 300, 1100
    f = key_profile(kind, Sk)
    qspec = ([(800, Sq)], 1) if causal else None
    kspec = ([(0, Sk)], 1) if causal else None
    o, l, q, k, v, scale = run_partial(1, 2, Sq, Sk, D, qspec, kspec, seed=11, k_row_scale=f)
    s = np.einsum("bqhd,bkhd->bhqk", q, k) * scale / math.log(2.0)  # log2 units
    if causal:
        s = np.where(positions(kspec)[None, None, None, :] <= positions(qspec)[None, None, :, None],
                     s, -np.inf)
    climb = s.max(axis=-1) - s[..., :128].max(axis=-1)
    if kind != "falling":
        assert (climb > 11.0).mean() > 0.5, "inputs do not reach the slow path"
    ro, rl = oracle.attention(q, k, v, scale, causal,
                              positions(qspec) if causal else None,
                              positions(kspec) if causal else None)
    check_attention(o, l, ro, rl, f"{kind} causal={causal} D={D}")


def test_bounded_wait_runs_out_then_context_usable(monkeypatch):
    """The failure path of the bounded device waits, without a fault: with the test hook
    USP_TEST_WITHHOLD_LOADS=1 the kernel's producer issues no loads, so every other role's wait
    runs out after USP_WAIT_BUDGET_MS; all roles stop and free their tensor memory, nothing is
    written outside the outputs, and usp_check_status reports USP_ERR_TIMEOUT.  The same context
    then computes the next call correctly."""
    t = torch()
    B, H, Sq, Sk, D = 1, 2, 300, 400, 128
    q = to_dev_bf16(synth.make_tensor_bits(3, 0, B, Sq, H, D))
    k = to_dev_bf16(synth.make_tensor_bits(3, 1, B, Sk, H, D))
    v = to_dev_bf16(synth.make_tensor_bits(3, 2, B, Sk, H, D))
    o = Guarded((B, Sq, H, D), t.float32)
    lse = Guarded((B, Sq, H), t.float32)
    status = t.zeros(1, dtype=t.int32, device="cuda")
    monkeypatch.setenv("USP_WAIT_BUDGET_MS", "50")
    monkeypatch.setenv("USP_TEST_WITHHOLD_LOADS", "1")
    t0 = time.monotonic()
    usp.usp_attn_partial(q, k, v, B, H, Sq, Sk, D, H * D, H * D, 1.0 / math.sqrt(D), o.view, lse.view,
                         status=status)
    assert usp.usp_check_status(status) == usp.USP_ERR_TIMEOUT
    assert time.monotonic() - t0 < 10.0
    o.check()
    lse.check()
    monkeypatch.delenv("USP_TEST_WITHHOLD_LOADS")
    monkeypatch.delenv("USP_WAIT_BUDGET_MS")
    assert usp.usp_check_status(status) == usp.USP_OK  # cleared by the previous check
    o2, l2, q2, k2, v2, scale = run_partial(B, H, Sq, Sk, D, seed=3)
    ro, rl = oracle.attention(q2, k2, v2, scale)
    check_attention(o2, l2, ro, rl, "after a timed-out call")
