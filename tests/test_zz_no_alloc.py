"""usp_attention_noalloc: usp_attention for callers that cannot allocate device memory (a host
application that owns every device allocation, or a path that cannot afford cudaMalloc's implicit
synchronisation).  It runs on a 128 MiB scratch array built into the library instead of a
workspace.

This file is named to be collected last, so that a run stopping at its first failure has run every
other test before these.  The GPU test calls the entry point through the C ABI four times in a
row on different problems and checks each result element by element against the fp64 oracle at
the parity tests' tolerances.  The first two calls run the ring steps separately, so their fp32
partials live in the shared scratch: the second call is causal with another ordering and grid, and
its fully masked chunk pairs leave partial slots that it must not read, so anything it picked up
from the first call's leftovers would show in its result.  The third call runs the fused ring,
the fourth a fused ring with its last blocks split into ring steps (their partials in the
scratch)."""
import math

import numpy as np
import pytest

import oracle
from sequence_attention_tcgen05_gb300 import build, synth, usp

O_MAX_ABS, O_MEAN_ABS, LSE_MAX_ABS = 2e-2, 2e-3, 1e-3


def _call_and_check(t, B, S, H, D, U, R, causal, order, out_dtype, seed):
    qb, kb, vb = synth.make_qkv_bits(B, S, H, D, seed)
    q, k, v = (t.from_numpy(x.view(np.int16)).view(t.bfloat16).cuda() for x in (qb, kb, vb))
    o = t.full((B, S, H, D), float("nan"), dtype=out_dtype, device="cuda")
    lse = t.full((B, S, H), float("nan"), dtype=t.float32, device="cuda")
    status = t.full((1,), 7, dtype=t.int32, device="cuda")
    usp.usp_attention_noalloc(q, k, v, B, S, H, D, 1.0 / math.sqrt(D), causal, U, R, o, lse,
                              order=order, status=status)
    assert usp.usp_check_status(status) == usp.USP_OK
    ref_o, ref_l = oracle.attention(oracle.widen_bf16(qb), oracle.widen_bf16(kb),
                                    oracle.widen_bf16(vb), 1.0 / math.sqrt(D), causal)
    got_o = o.float().cpu().numpy().astype(np.float64)
    got_l = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got_o))
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(got_l), fin)
    err = np.abs(got_o - ref_o)
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (err.max(), err.mean())
    assert np.abs(got_l[fin] - ref_l[fin]).max() <= LSE_MAX_ABS


@pytest.mark.gpu
def test_noalloc_matches_oracle_four_calls(monkeypatch):
    import torch as t
    build.build_library()
    monkeypatch.setenv("USP_RING_MERGE", "separate")
    # ring of 3, contiguous, non-causal, fp32 out: every partial slot written
    _call_and_check(t, 1, 1000, 4, 64, 1, 3, False, "contiguous", t.float32, seed=1)
    # Ulysses 2 x ring 2, stripe, causal, bf16 out, other shapes: masked pairs leave slots unread
    _call_and_check(t, 1, 777, 6, 128, 2, 2, True, "stripe", t.bfloat16, seed=2)
    monkeypatch.setenv("USP_RING_MERGE", "fused")
    # ring of 4, zigzag, causal, fp32 out, fused ring steps
    _call_and_check(t, 2, 600, 3, 128, 1, 4, True, "zigzag", t.float32, seed=3)
    # Ulysses 2 x ring 2, contiguous, non-causal, bf16 out: the last 2 blocks of the last ring
    # chunk run as separate ring steps, merged from the scratch
    monkeypatch.setenv("USP_RING_SPLIT", "2")
    _call_and_check(t, 1, 1537, 4, 128, 2, 2, False, "contiguous", t.bfloat16, seed=4)


def test_noalloc_rejects_problems_beyond_the_scratch(monkeypatch):
    """A 64K-token causal zigzag ring of 8 run with separate ring steps needs 8 fp32 partial
    slots of O (8.6 GB): rejected before any launch.  With the ring steps fused it needs only the
    status word, also when its half-chunks are not whole 128-row tiles (65535 tokens)."""
    build.build_library()
    L = usp.lib()
    monkeypatch.setenv("USP_RING_MERGE", "separate")
    st = L.usp_attention_noalloc(256, 256, 256, 1, 65535, 32, 128, 0.08, 1, 1, 8, None, None, 1,
                                 256, usp.USP_FP32, 256, None, None)
    assert st == usp.USP_ERR_WORKSPACE
    msg = L.usp_last_error().decode()
    assert "128 MiB" in msg and "needs" in msg
    monkeypatch.setenv("USP_RING_MERGE", "fused")
    assert usp.usp_attention_workspace_size(1, 65535, 32, 128, 1, 8, "zigzag", causal=True) == 256
