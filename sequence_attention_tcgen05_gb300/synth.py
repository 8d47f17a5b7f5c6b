"""Seeded synthetic inputs, shared by the CUDA path's tests and benchmark and by the oracle's tests.

This module holds no attention arithmetic. It has two parts:

* a counter-based generator: the SplitMix64 output function (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014) applied to a Weyl
  sequence, turned into N(0, 1) samples by the Box-Muller transform (Box and Muller,
  1958) and rounded to bfloat16 with round-to-nearest-even;
* the workload shapes of the pages' context-parallel runs (diffusion-transformer joint
  attention for FLUX.1-dev and Qwen-Image, and a long-context causal LLM), as plain data.

Element ``e`` of stream ``s`` under seed ``seed`` depends only on ``(seed, s, e)``, so any
element can be regenerated on its own and a sample of a huge tensor costs only that sample.
Box-Muller consumes the 64-bit words ``2j+1`` and ``2j+2`` of the stream for the element pair
``(2j, 2j+1)``: ``u1 = (w1 >> 11 + 1) 2^-53`` in (0, 1], ``u2 = (w2 >> 11) 2^-53`` in [0, 1),
``r = sqrt(-2 ln u1)``, element ``2j = r cos(2 pi u2)`` and ``2j+1 = r sin(2 pi u2)``, computed in
float64 and rounded to float32.  The bfloat16 input is the float32 sample rounded to nearest
even.  Streams: Q = 0, K = 1, V = 2; tensors are filled in row-major ``[B][S][H][D]`` order.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # elements per worker task

STREAM_Q, STREAM_K, STREAM_V = 0, 1, 2


def splitmix64_mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _stream_key(seed: int, stream: int) -> np.uint64:
    base = (np.uint64(seed & 0xFFFFFFFFFFFFFFFF) ^ (np.uint64(stream & 0xFFFFFFFF) << np.uint64(32)))
    return splitmix64_mix(np.array([base], dtype=np.uint64))[0]


def _words(key: np.uint64, idx: np.ndarray) -> np.ndarray:
    # Weyl sequence key + (idx + 1) * golden, mixed.
    with np.errstate(over="ignore"):
        x = key + (idx.astype(np.uint64) + np.uint64(1)) * _GOLDEN
    return splitmix64_mix(x)


def normal_f32_at(seed: int, stream: int, elems: np.ndarray) -> np.ndarray:
    """float32 N(0, 1) samples for arbitrary element indices of one stream."""
    elems = np.asarray(elems, dtype=np.int64)
    key = _stream_key(seed, stream)
    pair = elems >> 1
    w1 = _words(key, 2 * pair)
    w2 = _words(key, 2 * pair + 1)
    u1 = ((w1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (w2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u1))
    theta = 2.0 * np.pi * u2
    z = np.where((elems & 1) == 0, r * np.cos(theta), r * np.sin(theta))
    return z.astype(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest even); returns the raw uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = ((u + rounding) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _fill(seed: int, stream: int, n: int, workers: int | None = None) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    starts = list(range(0, n, _CHUNK))

    def work(s: int) -> None:
        e = min(n, s + _CHUNK)
        out[s:e] = normal_f32_at(seed, stream, np.arange(s, e, dtype=np.int64))

    if len(starts) == 1:
        work(0)
    else:
        with ThreadPoolExecutor(max_workers=workers or min(32, os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    return out


def make_tensor_bits(seed: int, stream: int, B: int, S: int, H: int, D: int,
                     text_rows: int = 0, text_scale: float = 1.0) -> np.ndarray:
    """One bf16 tensor ``[B][S][H][D]`` as uint16 bits.

    Rows ``t < text_rows`` of every batch are multiplied by ``text_scale`` in float32 before the
    rounding to bf16 (the joint text + image token layout: text tokens first)."""
    x = _fill(seed, stream, B * S * H * D).reshape(B, S, H, D)
    if text_rows and text_scale != 1.0:
        x[:, :text_rows] *= np.float32(text_scale)
    return bf16_bits(x)


def make_qkv_bits(B: int, S: int, H: int, D: int, seed: int = 0, text_rows: int = 0,
                  text_scale: float = 1.0):
    """Q, K, V bf16 bit tensors ``[B][S][H][D]`` (uint16), streams 0, 1, 2."""
    return tuple(make_tensor_bits(seed, s, B, S, H, D, text_rows, text_scale)
                 for s in (STREAM_Q, STREAM_K, STREAM_V))


def qkv_rows_bits(seed: int, stream: int, B: int, S: int, H: int, D: int,
                  b: int, t: np.ndarray, h: int, text_rows: int = 0,
                  text_scale: float = 1.0) -> np.ndarray:
    """Rows ``[len(t)][D]`` of head ``h``, batch ``b`` of one tensor, regenerated on their own."""
    t = np.asarray(t, dtype=np.int64)
    base = ((b * S + t) * H + h) * D
    elems = base[:, None] + np.arange(D, dtype=np.int64)[None, :]
    x = normal_f32_at(seed, stream, elems.ravel()).reshape(len(t), D)
    if text_rows and text_scale != 1.0:
        x[t < text_rows] *= np.float32(text_scale)
    return bf16_bits(x)


# ----------------------------------------------------------------------------------------------
# Workloads.  Shapes follow the pages' runs: FLUX.1-dev at 1024x1024 (512 text + 4096 image
# tokens) and 1008x1008 (512 + 3969), Qwen-Image at 1328x1328 (256 + 6889), 24 heads of 128;
# and a long-context causal LLM ring (32 heads of 128, 64K tokens, zigzag order).
# ----------------------------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    D: int
    S: int
    ulysses_degree: int
    ring_degree: int
    causal: bool = False
    order: str = "contiguous"      # contiguous | zigzag | stripe
    text_rows: int = 0
    text_scale: float = 1.0
    seq_lens: tuple = field(default=())   # per virtual rank; () = default split
    seed: int = 0

    @property
    def P(self) -> int:
        return self.ulysses_degree * self.ring_degree

    def attention_flops(self) -> float:
        """4 B H D x (number of unmasked query/key pairs)."""
        pairs = self.S * (self.S + 1) // 2 if self.causal else self.S * self.S
        return 4.0 * self.B * self.H * self.D * pairs


WORKLOADS = {
    "tiny_ring3": Workload("tiny_ring3", 1, 4, 64, 1000, 1, 3, seq_lens=(334, 333, 333)),
    "tiny_uaa3": Workload("tiny_uaa3", 1, 4, 64, 1000, 3, 1, seq_lens=(334, 333, 333)),
    "flux_1024_u2": Workload("flux_1024_u2", 1, 24, 128, 4608, 2, 1, text_rows=512, text_scale=0.5),
    "flux_1008_uaa2": Workload("flux_1008_uaa2", 1, 24, 128, 4481, 2, 1, seq_lens=(2241, 2240)),
    "flux_1008_uaa3": Workload("flux_1008_uaa3", 1, 24, 128, 4481, 3, 1, seq_lens=(1494, 1494, 1493)),
    "qwen_1328_u2r2": Workload("qwen_1328_u2r2", 1, 24, 128, 7145, 2, 2),
    "llm_64k_ring8_zigzag": Workload("llm_64k_ring8_zigzag", 1, 32, 128, 65536, 1, 8,
                                     causal=True, order="zigzag"),
    # The long-context ring at a quarter of the length (16 half-chunks of 1024 rows), small enough
    # for a full profiler capture of the attention kernel (402 MB of inputs, more than L2).
    "llm_16k_ring8_zigzag": Workload("llm_16k_ring8_zigzag", 1, 32, 128, 16384, 1, 8,
                                     causal=True, order="zigzag"),
    # Ring Anything / Ulysses Anything at large, uneven sizes: a sequence that no ring or head
    # count divides (zigzag half-chunks of 4111 and 4112 rows, not whole 128-row tiles), an uneven
    # stripe ring, and 24 heads over 5 Ulysses ranks (5/5/5/5/4 heads, 922/922/922/921/921 rows).
    "llm_64k257_ring8_zigzag": Workload("llm_64k257_ring8_zigzag", 1, 32, 128, 65793, 1, 8,
                                        causal=True, order="zigzag"),
    "llm_32k_ring4_stripe": Workload("llm_32k_ring4_stripe", 1, 32, 128, 32771, 1, 4,
                                     causal=True, order="stripe"),
    "flux_1024_uaa5": Workload("flux_1024_uaa5", 1, 24, 128, 4608, 5, 1, text_rows=512,
                               text_scale=0.5),
}
