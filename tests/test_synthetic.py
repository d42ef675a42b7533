"""The seeded input generators that feed both the oracle and the CUDA path: bf16 rounding
against torch's own conversion, determinism and thread-independence of the chunked streams,
the distributions' moments, and the layouts of the workloads (appended copies, shuffled
positions, needle rows, the decode cache's unwritten rows)."""
import numpy as np
import torch

from synthetic import (CONFIGS, DecodeConfig, bf16_bits, bf16_to_f32, make_decode, make_prefill,
                       normal_bf16, reduced, scale_offset)


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    g = np.random.default_rng(0)
    x = np.concatenate([g.standard_normal(100000).astype(np.float32) * 10.0 ** g.integers(-6, 6, 100000),
                        np.float32([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 0.0, 65504.0])])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bf16_bits(x), want)
    # the ties: 1 + 2^-8 rounds down to 1.0, 1 + 3 * 2^-8 up to 1 + 2^-6 (even mantissas)
    assert bf16_bits(np.float32([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert bf16_bits(np.float32([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82


def test_every_finite_bf16_pattern_round_trips_exactly():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = bf16_to_f32(bits)
    finite = np.isfinite(f)
    np.testing.assert_array_equal(bf16_bits(f[finite]), bits[finite])


def test_streams_are_deterministic_keyed_and_thread_independent():
    shape = (3, 1 << 21)  # 6 Mi elements: two keyed chunks
    a = normal_bf16(5, "k", shape, threads=1)
    np.testing.assert_array_equal(a, normal_bf16(5, "k", shape, threads=4))
    assert not np.array_equal(a, normal_bf16(5, "v", shape, threads=1))
    assert not np.array_equal(a, normal_bf16(6, "k", shape, threads=1))
    # the first chunk of a long tensor is the whole of a short one with the same key
    np.testing.assert_array_equal(a.reshape(-1)[:1000], normal_bf16(5, "k", (1000,)))


def test_moments_of_the_draws():
    x = bf16_to_f32(normal_bf16(9, "q_raw", (1 << 20,))).astype(np.float64)
    assert abs(x.mean()) < 0.005 and abs(x.std() - 1.0) < 0.005
    a, b = scale_offset(9, 64, 128)
    assert a.dtype == np.float32 and a.shape == (64, 128)
    assert abs(a.mean() - 1.0) < 0.01 and abs(a.std() - 0.1) < 0.01
    assert abs(b.mean()) < 0.01 and abs(b.std() - 0.1) < 0.01
    a2, _ = scale_offset(9, 64, 128, prefix="_c")
    assert not np.array_equal(a, a2)  # the copies' scale-offset is its own stream


def test_sft_layout_appended_copies_and_shuffled_positions():
    cfg = reduced(CONFIGS["sft_16k"], B=2, T=600, T_out=64)
    inp = make_prefill(cfg, 4)
    assert inp.q_raw.shape == (2, 664, 32, 128) and inp.qc_raw.shape == (2, 64, 32, 128)
    assert np.shares_memory(inp.qc_raw, inp.q_raw)  # the copies live at the tail of one buffer
    for bb in range(2):
        np.testing.assert_array_equal(np.sort(inp.pos[bb]), np.arange(536, 600))
    assert not np.array_equal(inp.pos[0], np.arange(536, 600))  # shuffled


def test_needle_rows_are_scaled_exactly():
    cfg = reduced(CONFIGS["prefill_1m"], T=4096, needle_frac=0.002)
    inp = make_prefill(cfg, 5)
    plain = normal_bf16(5, "k", (cfg.B, cfg.T, cfg.Hkv, cfg.d))
    assert inp.needles.size == round(0.002 * 4096)
    np.testing.assert_array_equal(bf16_to_f32(inp.k[:, inp.needles]), 4.0 * bf16_to_f32(plain[:, inp.needles]))
    rest = np.setdiff1d(np.arange(cfg.T), inp.needles)
    np.testing.assert_array_equal(inp.k[:, rest], plain[:, rest])


def test_decode_cache_rows_never_written_hold_nan():
    cfg = DecodeConfig("t", B=2, T0=50, steps=3, Hq=4, Hkv=2, d=16)
    inp = make_decode(cfg, 3)
    assert (inp.cache_len == 50).all()
    assert np.isnan(bf16_to_f32(inp.k_cache[:, 50:])).all() and np.isnan(bf16_to_f32(inp.v_cache[:, 50:])).all()
    assert np.isfinite(bf16_to_f32(inp.k_cache[:, :50])).all()
    assert inp.q_new.shape == (3, 2, 4, 16) and inp.k_new.shape == (3, 2, 2, 16)
