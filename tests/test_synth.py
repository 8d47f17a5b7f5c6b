"""The seeded input generator: determinism, sampling consistency, distribution, bf16 rounding."""
import numpy as np
import torch

from sequence_attention_tcgen05_gb300 import synth


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    # (state += golden; then the output function) are well known test vectors.
    g = np.uint64(0x9E3779B97F4A7C15)
    with np.errstate(over="ignore"):
        states = np.array([g, g * np.uint64(2), g * np.uint64(3)], dtype=np.uint64)
    out = synth.splitmix64_mix(states)
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_sampleable():
    q1 = synth.make_tensor_bits(0, synth.STREAM_K, 2, 9, 3, 8, text_rows=3, text_scale=0.5)
    q2 = synth.make_tensor_bits(0, synth.STREAM_K, 2, 9, 3, 8, text_rows=3, text_scale=0.5)
    assert np.array_equal(q1, q2)
    rows = np.array([0, 2, 3, 8])
    s = synth.qkv_rows_bits(0, synth.STREAM_K, 2, 9, 3, 8, b=1, t=rows, h=2, text_rows=3,
                            text_scale=0.5)
    assert np.array_equal(s, q1[1, rows, 2, :])
    other = synth.make_tensor_bits(1, synth.STREAM_K, 2, 9, 3, 8)
    assert not np.array_equal(other, synth.make_tensor_bits(0, synth.STREAM_K, 2, 9, 3, 8))


def test_normal_moments():
    z = synth.normal_f32_at(0, 0, np.arange(400000)).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert abs(((z > 1.0).mean()) - 0.158655) < 0.005


def test_bf16_rounding_matches_torch():
    x = synth.normal_f32_at(3, 1, np.arange(100000)) * np.float32(7.3)
    x = np.concatenate([x, np.array([0.0, -0.0, 1.0, 3.0e38, -1e-40], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.bf16_bits(x), ref)
    assert np.array_equal(synth.bf16_to_f32(ref), torch.from_numpy(ref.view(np.int16)).view(
        torch.bfloat16).float().numpy())


def test_workload_table():
    w = synth.WORKLOADS
    assert w["flux_1008_uaa3"].seq_lens == (1494, 1494, 1493)
    assert w["llm_64k_ring8_zigzag"].P == 8
    assert abs(w["flux_1024_u2"].attention_flops() - 4 * 24 * 128 * 4608 ** 2) < 1
