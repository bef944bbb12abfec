"""Pins of the oracle's f16 KV cache (each cached K and V element rounded to
the nearest IEEE binary16, ties to even, as it enters the cache) against
numpy's float16 conversion: layer 0's rows depend only on the token and the
position, so the f16 oracle's layer-0 cache must be exactly the f32
oracle's layer-0 rows rounded by numpy; loaded rows are rounded the same
way; and with the switch off nothing changes."""
import numpy as np

import oracle
import synth


def run(kv_f16, ids):
    model = synth.make_model(synth.TINY, 3)
    om = oracle.OracleModel(model, len(ids) + 1, kv_f16=kv_f16)
    om.prefill(ids)
    return om, model


def test_layer0_rows_are_the_f32_rows_rounded_to_f16():
    ids = synth.token_ids(1000, 2, 9, synth.TINY.vocab)
    o32, m32 = run(False, ids)
    o16, m16 = run(True, ids)
    for pos in range(len(ids)):
        k32, v32 = o32.kv_row(0, pos)
        k16, v16 = o16.kv_row(0, pos)
        assert np.array_equal(k16, np.float16(k32).astype(np.float64)), pos
        assert np.array_equal(v16, np.float16(v32).astype(np.float64)), pos
        assert not np.array_equal(k16, k32)  # the rounding did something


def test_every_cached_element_is_an_f16_value():
    ids = synth.token_ids(1000, 4, 7, synth.TINY.vocab)
    o16, _ = run(True, ids)
    for layer in range(synth.TINY.n_layers):
        for pos in range(len(ids)):
            k, v = o16.kv_row(layer, pos)
            assert np.array_equal(np.float16(k).astype(np.float64), k)
            assert np.array_equal(np.float16(v).astype(np.float64), v)


def test_loaded_rows_are_rounded():
    cfg = synth.TINY
    model = synth.make_model(cfg, 0)
    k, v = synth.kv_fill(cfg, 5, 0, 6)
    o16 = oracle.OracleModel(model, 8, kv_f16=True)
    o16.kv_load(k, v)
    o32 = oracle.OracleModel(model, 8)
    o32.kv_load(k, v)
    for layer in range(cfg.n_layers):
        for pos in range(6):
            a, b = o16.kv_row(layer, pos)
            c, d = o32.kv_row(layer, pos)
            assert np.array_equal(a, np.float16(k[layer, pos]).astype(np.float64))
            assert np.array_equal(b, np.float16(v[layer, pos]).astype(np.float64))
            assert np.array_equal(c, k[layer, pos].astype(np.float64))
            assert np.array_equal(d, v[layer, pos].astype(np.float64))


def test_the_rounding_moves_the_logits_only_slightly():
    ids = synth.token_ids(1000, 6, 12, synth.TINY.vocab)
    model = synth.make_model(synth.TINY, 3)
    _, l32 = oracle.OracleModel(model, 16).prefill(ids)
    _, l16 = oracle.OracleModel(model, 16, kv_f16=True).prefill(ids)
    d = float(np.max(np.abs(l16 - l32)))
    assert 0.0 < d < 2e-3 * float(np.max(np.abs(l32)))
