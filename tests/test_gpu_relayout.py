"""GPU re-layout and reorder kernels against the oracle's index loops: bit-exact."""
import numpy as np
import pytest

import oracle
from sequence_attention_tcgen05_gb300 import usp

from gpu_util import Guarded, bits_of, torch

pytestmark = pytest.mark.gpu


def _dev(arr_u16_or_u32):
    t = torch()
    if arr_u16_or_u32.dtype == np.uint16:
        return t.from_numpy(arr_u16_or_u32.view(np.int16).copy()).view(t.bfloat16).cuda()
    return t.from_numpy(arr_u16_or_u32.view(np.float32).copy()).cuda()


CASES = [  # B, H, D, seq_lens, head_counts
    (1, 24, 128, [2304, 2304], None),          # FLUX 1024^2, Ulysses 2
    (1, 24, 128, [2241, 2240], None),          # FLUX 1008^2, UAA 2
    (1, 24, 128, [1494, 1494, 1493], None),    # FLUX 1008^2, UAA 3
    (1, 4, 64, [334, 333, 333], [2, 1, 1]),    # tiny, uneven heads
    (2, 5, 64, [7, 0, 13, 1], [2, 1, 1, 1]),   # empty chunk, 1-token chunk, B = 2
    (3, 6, 8, [5, 9], [3, 3]),                 # small D: narrower vectors
]


@pytest.mark.parametrize("B,H,D,lens,heads", CASES)
@pytest.mark.parametrize("elem", ["bf16", "fp32"])
def test_seq2head_head2seq_bit_exact(B, H, D, lens, heads, elem):
    rng = np.random.default_rng(7)
    S = sum(lens)
    n = B * S * H * D
    src = rng.integers(0, 2**16 if elem == "bf16" else 2**32, size=n, dtype=np.uint64)
    src = src.astype(np.uint16 if elem == "bf16" else np.uint32)
    if elem == "fp32":
        src &= np.uint32(0x7F7FFFFF)  # finite patterns: torch.fill etc. keep bits anyway
    want = oracle.seq2head(src, B, H, D, lens, heads)
    x = _dev(src)
    y = Guarded((n,), x.dtype)
    usp.usp_relayout_seq2head(x, y.view, B, H, D, lens, heads)
    torch().cuda.synchronize()
    y.check()
    assert np.array_equal(bits_of(y.view), want)
    back = Guarded((n,), x.dtype)
    usp.usp_relayout_head2seq(y.view, back.view, B, H, D, lens, heads)
    torch().cuda.synchronize()
    back.check()
    assert np.array_equal(bits_of(back.view), src)
    assert np.array_equal(oracle.head2seq(want, B, H, D, lens, heads), src)


def test_lse_head2seq_d1():
    B, H, lens, heads = 1, 24, [2241, 2240], [12, 12]
    S = sum(lens)
    src = np.random.default_rng(3).standard_normal(B * S * H).astype(np.float32)
    x = _dev(src.view(np.uint32))
    y = Guarded((B * S * H,), x.dtype)
    usp.usp_relayout_head2seq(x, y.view, B, H, 1, lens, heads)
    torch().cuda.synchronize()
    y.check()
    assert np.array_equal(bits_of(y.view), oracle.head2seq(src, B, H, 1, lens, heads).view(np.uint32))


@pytest.mark.parametrize("order", ["contiguous", "zigzag", "stripe"])
@pytest.mark.parametrize("B,S,H,D,R", [(1, 1000, 4, 64, 3), (2, 517, 3, 128, 4), (1, 4096, 2, 128, 8)])
def test_reorder_bit_exact(order, B, S, H, D, R):
    rng = np.random.default_rng(11)
    src = rng.integers(0, 2**16, size=(B, S, H, D), dtype=np.uint64).astype(np.uint16)
    pos = oracle.ring_positions(order, S, R)
    want = np.concatenate([src[:, p].reshape(-1) for p in pos])
    x = _dev(src.reshape(-1))
    y = Guarded((src.size,), x.dtype)
    usp.usp_reorder(x, y.view, B, S, H, D, R, order)
    torch().cuda.synchronize()
    y.check()
    assert np.array_equal(bits_of(y.view), want)
    back = Guarded((src.size,), x.dtype)
    usp.usp_reorder(y.view, back.view, B, S, H, D, R, order, inverse=True)
    torch().cuda.synchronize()
    back.check()
    assert np.array_equal(bits_of(back.view), src.reshape(-1))


@pytest.mark.parametrize("B,H,D,lens,heads", [CASES[1], CASES[2], CASES[4]])
def test_multi_tensor_relayout_bit_exact(B, H, D, lens, heads):
    """Q, K, V in one launch (usp_relayout_seq2head_multi) and back (head2seq_multi): each tensor
    bit-exact against the oracle's index loops, as if re-laid on its own."""
    rng = np.random.default_rng(5)
    S = sum(lens)
    n = B * S * H * D
    srcs = [rng.integers(0, 2**16, size=n, dtype=np.uint64).astype(np.uint16) for _ in range(3)]
    xs = [_dev(x) for x in srcs]
    ys = [Guarded((n,), xs[0].dtype) for _ in range(3)]
    usp.usp_relayout_seq2head_multi(xs, [y.view for y in ys], B, H, D, lens, heads)
    torch().cuda.synchronize()
    for src, y in zip(srcs, ys):
        y.check()
        assert np.array_equal(bits_of(y.view), oracle.seq2head(src, B, H, D, lens, heads))
    backs = [Guarded((n,), xs[0].dtype) for _ in range(3)]
    usp.usp_relayout_head2seq_multi([y.view for y in ys], [b.view for b in backs], B, H, D, lens,
                                    heads)
    torch().cuda.synchronize()
    for src, b in zip(srcs, backs):
        b.check()
        assert np.array_equal(bits_of(b.view), src)
