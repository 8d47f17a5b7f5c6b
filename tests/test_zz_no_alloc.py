"""usp_attention_noalloc: usp_attention for callers that cannot allocate device memory (a host
application that owns every device allocation, or a path that cannot afford cudaMalloc's implicit
synchronisation).  It runs on a 128 MiB scratch array built into the library instead of a
workspace.

This file is named to be collected last, so that a run stopping at its first failure has run every
other test before these.  The GPU test calls the entry point through the C ABI twice in a row, on
two different problems, and checks each result against usp_attention with a torch-allocated
workspace, within the tolerances the parity tests use; the second call also shows that the first
call's leftovers in the shared scratch do not leak into the next result."""
import math

import numpy as np
import pytest

from sequence_attention_tcgen05_gb300 import build, synth, usp


def _run_pair(t, B, S, H, D, U, R, causal, order, out_dtype, seed):
    qb, kb, vb = synth.make_qkv_bits(B, S, H, D, seed)
    q, k, v = (t.from_numpy(x.view(np.int16)).view(t.bfloat16).cuda() for x in (qb, kb, vb))
    ref_o, ref_l = usp.attention(q, k, v, causal=causal, ulysses_degree=U, ring_degree=R,
                                 order=order, out_dtype=out_dtype)
    o = t.full((B, S, H, D), float("nan"), dtype=out_dtype, device="cuda")
    lse = t.full((B, S, H), float("nan"), dtype=t.float32, device="cuda")
    status = t.full((1,), 7, dtype=t.int32, device="cuda")
    usp.usp_attention_noalloc(q, k, v, B, S, H, D, 1.0 / math.sqrt(D), causal, U, R, o, lse,
                              order=order, status=status)
    assert usp.usp_check_status(status) == usp.USP_OK
    t.cuda.synchronize()
    d_o = (o.float() - ref_o.float()).abs()
    fin = t.isfinite(ref_l)
    assert bool((t.isfinite(lse) == fin).all())
    assert float(d_o.max()) <= 2e-2 and float(d_o.mean()) <= 2e-3
    assert float((lse[fin] - ref_l[fin]).abs().max()) <= 1e-3
    return float(d_o.max())


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    import torch as t
    build.build_library()
    # ring of 3, causal, zigzag, fp32 out; then Ulysses 2 x ring 2, non-causal, bf16 out
    e1 = _run_pair(t, 1, 1000, 4, 64, 1, 3, True, "zigzag", t.float32, seed=1)
    e2 = _run_pair(t, 1, 777, 6, 128, 2, 2, False, "contiguous", t.bfloat16, seed=2)
    assert e1 == 0.0 and e2 == 0.0  # same kernels on the same inputs: identical results


def test_noalloc_rejects_problems_beyond_the_scratch():
    """FLUX-sized ring-2 fp32 output needs far more than 128 MiB: rejected before any launch."""
    build.build_library()
    L = usp.lib()
    st = L.usp_attention_noalloc(256, 256, 256, 1, 65536, 32, 128, 0.08, 1, 1, 8, None, None, 1,
                                 256, usp.USP_FP32, 256, None, None)
    assert st == usp.USP_ERR_WORKSPACE
    msg = L.usp_last_error().decode()
    assert "128 MiB" in msg and "needs" in msg
