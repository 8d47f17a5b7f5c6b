"""Helpers for the GPU parity tests: device copies of the seeded inputs, guard-banded outputs
(canaries instead of a sanitizer) and the tolerance checks."""
import numpy as np

import oracle

# Tolerances for bf16 inputs with fp32 accumulation against the fp64 oracle.
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3

GUARD = 4096  # elements of canary on each side of an output
SENTINEL_F32 = np.float32(1.2345e30)


def torch():
    import torch as t
    return t


def to_dev_bf16(bits: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(t.bfloat16).cuda()


def bits_of(x) -> np.ndarray:
    t = torch()
    if x.dtype == t.bfloat16:
        return x.view(t.int16).cpu().numpy().view(np.uint16)
    return x.cpu().numpy().view(np.uint32)


class Guarded:
    """A device buffer with canaries before and after the visible part."""

    def __init__(self, shape, dtype):
        t = torch()
        n = int(np.prod(shape))
        self.n = n
        self.full = t.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
        if dtype == t.bfloat16:
            self.full.view(t.int16).fill_(0x7F7F)
        else:
            self.full.fill_(float(SENTINEL_F32))
        self.view = self.full[GUARD:GUARD + n].view(*shape)

    def check(self):
        t = torch()
        head, tail = self.full[:GUARD], self.full[GUARD + self.n:]
        if self.full.dtype == t.bfloat16:
            ok = bool((head.view(t.int16) == 0x7F7F).all()) and bool((tail.view(t.int16) == 0x7F7F).all())
        else:
            ok = bool((head == float(SENTINEL_F32)).all()) and bool((tail == float(SENTINEL_F32)).all())
        assert ok, "write outside the output buffer"


def check_attention(o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray,
                    tag: str = ""):
    o_gpu = o_gpu.astype(np.float64)
    lse_gpu = lse_gpu.astype(np.float64)
    assert o_gpu.shape == o_ref.shape, tag
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin), f"{tag}: -inf pattern of lse differs"
    assert np.all(lse_gpu[~fin] == -np.inf), tag
    err = np.abs(o_gpu - o_ref)
    assert np.all(np.isfinite(o_gpu)), f"{tag}: non-finite output"
    assert err.max() <= O_MAX_ABS, f"{tag}: O max abs err {err.max():.3e}"
    assert err.mean() <= O_MEAN_ABS, f"{tag}: O mean abs err {err.mean():.3e}"
    lerr = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    assert lerr <= LSE_MAX_ABS, f"{tag}: LSE max abs err {lerr:.3e}"
    # shown with pytest -s: the measured errors next to the tolerances
    print(f"[parity] {tag}: O max abs {err.max():.3e} mean abs {err.mean():.3e}, LSE max abs {lerr:.3e}")
    return float(err.max()), float(err.mean())


def widen(bits):
    return oracle.widen_bf16(bits)
