"""Checks of the seeded input generator against independent restatements:
splitmix64 in pure Python, numpy's f16 rounding, torch's bf16 rounding, and
the Q8_0 quantiser's round-trip bound."""
import numpy as np
import pytest

import synth

M64 = (1 << 64) - 1


def py_mix64(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def py_stream(seed, t):
    return py_mix64(seed ^ ((0xD1B54A32D192ED03 * (t + 1)) & M64))


def py_draw(s, k):
    return py_mix64((s + (k + 1) * 0x9E3779B97F4A7C15) & M64)


def test_splitmix64_reference_values():
    # splitmix64 seeded with 0 (published first output 0xE220A8397B1DCDAF)
    assert py_mix64(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF
    L = synth.lib()
    for seed, t, k in [(0, 0, 0), (0, 5, 17), (1234567, 3, 99999), (2 ** 63 + 5, 70000, 3)]:
        s = L.tqs_stream(seed, t)
        assert s == py_stream(seed, t)
        assert L.tqs_draw(s, k) == py_draw(s, k)


def test_normal_draw_definition_and_moments():
    s = py_stream(0, 9)
    for i in [0, 1, 1000]:
        tot = 0
        for w in range(3):
            r = py_draw(s, 3 * i + w)
            tot += sum((r >> (16 * j)) & 0xFFFF for j in range(4))
        z = (2 * tot - 12 * 65535) / 131072.0
        assert synth.lib().tqs_std_normal(s, i) == z
    x = synth.normal_f32(0, 9, 2_000_000, 0.0, 0.02).astype(np.float64)
    assert abs(x.mean()) < 1e-4 and abs(x.std() - 0.02) < 1e-4
    assert np.abs(x).max() <= 6 * 0.02


def test_f16_encoding_matches_numpy_rounding():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 1e-3,
        rng.standard_normal(20000).astype(np.float32) * 1e3,
        (rng.random(20000) * 2 ** -14).astype(np.float32),  # subnormal range
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2 ** -25, 2 ** -25 * 1.0001,
                  2 ** -24 * 1.5, 2 ** -24 * 2.5, np.inf, -np.inf], dtype=np.float32),
    ])
    # halfway cases between adjacent f16 values
    h = np.arange(0x0400, 0x7BFF, 97, dtype=np.uint16).view(np.float16).astype(np.float32)
    h2 = (np.arange(0x0401, 0x7C00, 97, dtype=np.uint16)).view(np.float16).astype(np.float32)
    vals = np.concatenate([vals, (h + h2) / 2]).astype(np.float32)
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([synth.f32_to_f16_bits(v) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_encoding_matches_torch_rounding():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(20000).astype(np.float32) * s for s in (1e-30, 0.02, 1e20)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([synth.f32_to_bf16_bits(v) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_q8_0_quantiser_round_trip_bound():
    rows, cols = 64, 256
    q = synth.q8_0_matrix(0, 3, rows, cols, 0.02)
    w = synth.normal_f32(0, 3, rows * cols, 0.0, 0.02).reshape(rows, cols)  # same stream
    blk = q.reshape(rows, cols // 32, 34)
    scale = blk[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    quants = blk[:, :, 2:].view(np.int8).astype(np.float64)
    wb = w.reshape(rows, cols // 32, 32).astype(np.float64)
    d = (np.abs(wb).max(axis=2).astype(np.float32) / np.float32(127)).astype(np.float64)
    err = np.abs(wb - scale[:, :, None] * quants)
    bound = d[:, :, None] * 0.5 * (1 + 1e-6) + np.abs(d - scale)[:, :, None] * 127
    assert np.all(err <= bound)
    # the largest magnitude of every block maps to +-127
    assert np.all(np.abs(quants).max(axis=2) == 127)
    assert np.all(quants >= -127)


def test_zero_block_and_token_ids():
    z = synth.quantize_rows(np.zeros((1, 32), dtype=np.float32))
    assert np.all(z == 0)
    ids = synth.token_ids(1000, 0, 511, 151936)
    assert ids.min() >= 0 and ids.max() < 151936
    assert np.array_equal(ids, synth.token_ids(1000, 0, 511, 151936))
    assert not np.array_equal(ids, synth.token_ids(1000, 1, 511, 151936))
    s = py_stream(1000, 0x10000)
    assert ids[3] == py_draw(s, 3) % 151936


def test_model_shapes():
    m = synth.make_model(synth.TINY, 0)
    cfg = synth.TINY
    assert m.lm_head.shape == (cfg.vocab, cfg.hidden // 32 * 34)
    d = m.layers[1]
    assert d["wq"].shape == (cfg.q_width, cfg.hidden // 32 * 34)
    assert d["wo"].shape == (cfg.hidden, cfg.q_width // 32 * 34)
    assert d["w_down"].shape == (cfg.hidden, cfg.intermediate // 32 * 34)
    assert d["q_norm"].shape == (cfg.head_dim,)
    b = synth.make_model(synth.ModelConfig(1, 64, 2, 1, 32, 96, 128, False, "bf16", 1e5), 0)
    assert b.layers[0]["wq"].dtype == np.uint16 and "q_norm" not in b.layers[0]
