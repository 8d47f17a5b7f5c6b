"""The bench's algorithmic counts (the numerators of every GB/s and TFLOP/s it reports) against
values derived by hand from the workload definitions; CPU only (the host planner needs no GPU)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sequence_attention_tcgen05_gb300 import build, synth  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build_library()


def test_attention_flops():
    w = synth.WORKLOADS
    assert w["flux_1024_u2"].attention_flops() == 4 * 24 * 128 * 4608 ** 2          # 260.92 G
    assert w["flux_1008_uaa2"].attention_flops() == 4 * 24 * 128 * 4481 ** 2        # 246.74 G
    assert w["qwen_1328_u2r2"].attention_flops() == 4 * 24 * 128 * 7145 ** 2        # 627.32 G
    # causal: every (query, key <= query) pair once, S (S + 1) / 2 of them
    assert w["llm_64k_ring8_zigzag"].attention_flops() == 4 * 32 * 128 * 65536 * 65537 // 2
    assert w["tiny_ring3"].attention_flops() == 4 * 4 * 64 * 1000 ** 2


def test_no_reorder_pass():
    # every workload's Q, K, V are addressed in place (zigzag 64K: a piece dimension over 16 equal
    # half-chunks of 4096; 65793 tokens, half-chunks of 4111/4112 rows: a span map per chunk), so
    # the step has no Q/K/V pass
    for w in synth.WORKLOADS.values():
        assert bench.phase_bytes(w, 2, "separate")["qkv_relayout"] == 0, w.name


def test_qwen_merge_bytes():
    # 7145 x 24 = 171480 (row, head) vectors; two fp32 partials of 128 + their LSEs read, bf16 O
    # and fp32 LSE written
    v = 7145 * 24
    expect = 2 * v * (128 * 4 + 4) + v * 128 * 2 + v * 4
    assert expect == 221552160
    assert bench.phase_bytes(synth.WORKLOADS["qwen_1328_u2r2"], 2, "separate")["merge"] == expect
    # fused ring steps have no merge pass
    assert bench.phase_bytes(synth.WORKLOADS["qwen_1328_u2r2"], 2, "fused")["merge"] == 0


def test_causal_zigzag_merge_bytes():
    # Zigzag, 8 ring ranks: rank r holds half-chunks r and 15 - r (4096 rows each), so its earliest
    # key is at 4096 r.  A query in half-chunk p therefore sees keys of min(p + 1, 8) ranks:
    # 1 + 2 + ... + 8 + 8 x 8 = 100 partials over the 16 half-chunks, 6.25 per vector on average.
    vectors = 65536 * 32
    seen = sum(min(p + 1, 8) for p in range(16)) * 4096 * 32
    assert seen * 8 == vectors * 50  # 6.25 = 50 / 8
    expect = 8 * vectors * 4 + seen * 128 * 4 + vectors * 128 * 2 + vectors * 4
    assert expect == 7323254784
    w = synth.WORKLOADS["llm_64k_ring8_zigzag"]
    assert bench.visible_partial_vectors(w) == seen
    assert bench.phase_bytes(w, 2, "separate")["merge"] == expect


def test_single_ring_rank_has_no_merge():
    for name in ("flux_1024_u2", "flux_1008_uaa2", "flux_1008_uaa3", "tiny_uaa3"):
        assert bench.phase_bytes(synth.WORKLOADS[name], 2, "none")["merge"] == 0


def test_roofline_peak_by_timed_length():
    """A timed region of at least SUSTAINED_MS of device time divides by the sustained bf16 peak,
    a shorter one by the burst peak."""
    peaks = {"bf16_tflops": 1842.5, "bf16_tflops_sustained": 1679.4, "hbm_gbs": 6791.4}
    assert bench.roofline_peak(peaks, 20 * 21.2) == (1679.4, True)      # 64K ring, 20 steps
    assert bench.roofline_peak(peaks, 100 * 0.167) == (1842.5, False)   # FLUX, 100 steps
    assert bench.roofline_peak(peaks, bench.SUSTAINED_MS) == (1679.4, True)


def test_kernel_hash_ignores_comments_and_whitespace():
    """The DRAM traffic recorded for the attention kernel stays valid across comment edits and is
    dropped when the code changes."""
    code = "int f(int x) {\n  // one\n  return x + 1; /* two\n lines */\n}\n"
    assert bench.code_of(code) == "intf(intx){returnx+1;}"
    assert bench.code_of(code.replace("// one", "// another comment")) == bench.code_of(code)
    assert bench.code_of(code.replace("x + 1", "x + 2")) != bench.code_of(code)
