"""Pins for the oracle: each check ties it to something other than itself —
numpy / scipy as independent decoders and contractions, closed forms,
invariants of the mathematics, brute force on tiny inputs, and the worked
cases of inferno.rs "IV.4: One command buffer per token", "The correctness
ladder"."""
import dataclasses
import math

import numpy as np
import pytest

import oracle
import synth
from tests.p1_lcg import P1Rng, random_q8_bytes

scipy_special = pytest.importorskip("scipy.special")


def np_dequant_q8_0(w: np.ndarray, cols: int) -> np.ndarray:
    """Independent Q8_0 decoder: numpy's float16 view of the two scale bytes
    times the int8 quants."""
    rows = w.size // (cols // 32 * 34)
    blk = np.ascontiguousarray(w, dtype=np.uint8).reshape(rows, cols // 32, 34)
    scales = blk[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    quants = blk[:, :, 2:].view(np.int8).astype(np.float64)
    return (scales[:, :, None] * quants).reshape(rows, cols)


def np_bf16(w: np.ndarray) -> np.ndarray:
    return (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------- formats

def test_f16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zero and subnormal edges
    assert math.copysign(1.0, oracle.f16_to_f64(0x8000)) == -1.0
    assert oracle.f16_to_f64(0x0001) == 2.0 ** -24
    assert oracle.f16_to_f64(0x3C00) == 1.0


def test_bf16_decode_patterns():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ref = np_bf16(bits)
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_q8_0_block_dequant_brute_force():
    """Every int8 quant against a spread of scales, including subnormal f16."""
    scales = [0x0001, 0x03FF, 0x0400, 0x2C00, 0x1234, 0x3C00, 0x7BFF, 0x8001, 0xAC00]
    for sb in scales:
        s = np.array([sb], dtype=np.uint16).view(np.float16).astype(np.float64)[0]
        for start in range(0, 256, 32):
            q = np.arange(start, start + 32, dtype=np.int32).astype(np.uint8)
            blk = np.concatenate([np.array([sb & 0xFF, sb >> 8], dtype=np.uint8), q])
            got = oracle.q8_0_dequant_block(blk)
            ref = s * q.view(np.int8).astype(np.float64)
            assert np.array_equal(got, ref)
            # the product is exact in f32 as well: 11-bit scale x 8-bit quant
            assert np.array_equal(got.astype(np.float32).astype(np.float64), got)


# ----------------------------------------------------------------- matvecs

def test_q8_0_matvec_exact_integer_case():
    """Power-of-two scales and small-integer x make the result an exact
    integer multiple of a power of two: compared for equality with int64."""
    rng = np.random.default_rng(5)
    rows, cols = 37, 256
    quants = rng.integers(-127, 128, size=(rows, cols // 32, 32))
    exps = rng.integers(-4, 4, size=(rows, cols // 32))
    sbits = (15 + exps).astype(np.uint16) << 10  # f16 of 2^e
    w = np.zeros((rows, cols // 32, 34), dtype=np.uint8)
    w[:, :, 0] = sbits & 0xFF
    w[:, :, 1] = sbits >> 8
    w[:, :, 2:] = quants.astype(np.int8).view(np.uint8)
    x = rng.integers(-8, 9, size=cols)
    got = oracle.q8_0_matvec(w.reshape(rows, -1), cols, x.astype(np.float64))
    # exact: sum_b 2^e_b * sum_j q x, scaled by 2^4 into integers
    ints = (quants * x.reshape(cols // 32, 32)[None]).sum(axis=2)  # [rows, blocks]
    ref16 = (ints * (2 ** (exps + 4))).sum(axis=1)
    assert np.array_equal(got * 16, ref16.astype(np.float64))


def test_q8_0_matvec_p1_case():
    """The matvec case of the correctness ladder: p=50 rows, n=96 columns,
    fabricated Q8 bytes (seed 7), x from the LCG (seed 42)."""
    p, n = 50, 96
    w = random_q8_bytes(p, n, 7)
    x = P1Rng(42).vec(n).astype(np.float64)
    ref = np_dequant_q8_0(w, n) @ x
    got = oracle.q8_0_matvec(w, n, x)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)
    # the fabricated scale is f16 0x2c00 = 0.0625
    assert oracle.f16_to_f64(0x2C00) == 0.0625


def test_q8_0_matvec_random_rows_and_layout():
    cfg = synth.TINY
    w = synth.q8_0_matrix(3, 77, 64, 256)
    x = synth.normal_f32(3, 78, 256).astype(np.float64)
    got = oracle.q8_0_matvec(w, 256, x)
    assert np.allclose(got, np_dequant_q8_0(w, 256) @ x, rtol=1e-12, atol=1e-14)
    # a transposed operand or a wrong block stride would not survive this
    assert cfg.hidden == 256


def test_bf16_matvec():
    w = synth.bf16_matrix(1, 9, 33, 96)
    x = synth.normal_f32(1, 10, 96).astype(np.float64)
    assert np.allclose(oracle.bf16_matvec(w, x), np_bf16(w) @ x, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_vector_closed_form():
    n, c, eps = 1024, 0.37, 1e-6
    g = synth.normal_f32(0, 1, n, 1.0, 0.1)
    out = oracle.rmsnorm(np.full(n, c), g, eps)
    ref = c / math.sqrt(c * c + eps) * g.astype(np.float64)
    assert np.allclose(out, ref, rtol=1e-14, atol=0)


def test_rmsnorm_invariants():
    rng = P1Rng(3)
    for rows, dim in [(1, 1024), (16, 128)]:
        x = rng.vec(rows * dim).astype(np.float64)
        g = np.ones(dim, dtype=np.float32)
        out = oracle.rmsnorm(x, g, 0.0).reshape(rows, dim)
        # unit mean square per row, direction preserved
        assert np.allclose((out ** 2).mean(axis=1), 1.0, rtol=1e-13)
        xr = x.reshape(rows, dim)
        assert np.allclose(out * np.sqrt((xr ** 2).mean(axis=1, keepdims=True)), xr, rtol=1e-12)
        # scale invariance with eps = 0, gain applied elementwise
        g2 = (rng.vec(dim) + np.float32(1.5)).astype(np.float32)
        a = oracle.rmsnorm(3.5 * x, g2, 0.0).reshape(rows, dim)
        assert np.allclose(a, out * g2.astype(np.float64), rtol=1e-12)


# ----------------------------------------------------------------- RoPE

def test_rope_half_split_pairing_and_frequency():
    # hd=4, theta=100: pair (0,2) turns at frequency 1, pair (1,3) at 100^-1/2 = 0.1
    pos = 10
    e0 = oracle.rope(np.array([1.0, 0, 0, 0]), 1, 4, pos, 100.0)
    assert np.allclose(e0, [math.cos(10), 0, math.sin(10), 0], atol=1e-15)
    e1 = oracle.rope(np.array([0, 1.0, 0, 0]), 1, 4, pos, 100.0)
    assert np.allclose(e1, [0, math.cos(1.0), 0, math.sin(1.0)], atol=1e-14)
    e3 = oracle.rope(np.array([0, 0, 0, 1.0]), 1, 4, pos, 100.0)
    assert np.allclose(e3, [0, -math.sin(1.0), 0, math.cos(1.0)], atol=1e-14)


def test_rope_invariants():
    rng = P1Rng(11)
    heads, hd, theta = 4, 16, 1e6
    x = rng.vec(heads * hd).astype(np.float64)
    # position 0 is the identity
    assert np.array_equal(oracle.rope(x, heads, hd, 0, theta), x)
    r = oracle.rope(x, heads, hd, 137, theta).reshape(heads, hd)
    xr = x.reshape(heads, hd)
    half = hd // 2
    # every rotated pair keeps its norm
    assert np.allclose(r[:, :half] ** 2 + r[:, half:] ** 2, xr[:, :half] ** 2 + xr[:, half:] ** 2,
                       rtol=1e-13)
    # R(p1) then R(p2) equals R(p1 + p2)
    two = oracle.rope(oracle.rope(x, heads, hd, 100, theta), heads, hd, 37, theta)
    assert np.allclose(two, r.reshape(-1), rtol=1e-11, atol=1e-12)
    # q(p) . k(p') depends on p - p' only
    q = rng.vec(hd).astype(np.float64)
    k = rng.vec(hd).astype(np.float64)
    d1 = oracle.rope(q, 1, hd, 500, theta) @ oracle.rope(k, 1, hd, 480, theta)
    d2 = oracle.rope(q, 1, hd, 20, theta) @ oracle.rope(k, 1, hd, 0, theta)
    assert abs(d1 - d2) < 1e-11


# ----------------------------------------------------------------- attention

def scipy_attention(q, K, V, nq, nkv, hd):
    out = np.zeros(nq * hd)
    g = nq // nkv
    for h in range(nq):
        kh = K[:, (h // g) * hd:(h // g + 1) * hd]
        vh = V[:, (h // g) * hd:(h // g + 1) * hd]
        a = scipy_special.softmax(kh @ q[h * hd:(h + 1) * hd] / math.sqrt(hd))
        out[h * hd:(h + 1) * hd] = a @ vh
    return out


def test_attention_p1_case():
    """4 query heads, 2 kv heads, head_dim 16, 9 cached rows (LCG seed 23)."""
    nq, nkv, hd, S = 4, 2, 16, 9
    rng = P1Rng(23)
    q = rng.vec(nq * hd).astype(np.float64)
    K = rng.vec(S * nkv * hd).astype(np.float64).reshape(S, nkv * hd)
    V = rng.vec(S * nkv * hd).astype(np.float64).reshape(S, nkv * hd)
    got = oracle.attention(q, K, V, nq, nkv, hd)
    assert np.allclose(got, scipy_attention(q, K, V, nq, nkv, hd), rtol=1e-13, atol=1e-14)


def test_attention_special_cases():
    nq, nkv, hd = 4, 2, 8
    rng = np.random.default_rng(0)
    q = rng.standard_normal(nq * hd)
    # one cached row: the output is that row's V exactly
    K1 = rng.standard_normal((1, nkv * hd))
    V1 = rng.standard_normal((1, nkv * hd))
    o = oracle.attention(q, K1, V1, nq, nkv, hd).reshape(nq, hd)
    for h in range(nq):
        assert np.array_equal(o[h], V1[0, (h // 2) * hd:(h // 2 + 1) * hd])
    # equal scores (q = 0): the mean of the V rows
    S = 7
    K = rng.standard_normal((S, nkv * hd))
    V = rng.standard_normal((S, nkv * hd))
    o = oracle.attention(np.zeros(nq * hd), K, V, nq, nkv, hd).reshape(nq, hd)
    assert np.allclose(o[1], V[:, 0:hd].mean(axis=0), rtol=1e-13)
    assert np.allclose(o[3], V[:, hd:2 * hd].mean(axis=0), rtol=1e-13)
    # one-hot V rows expose the softmax weights: positive, summing to one
    S = hd
    Voh = np.tile(np.eye(hd), (1, nkv))
    w = oracle.attention(q, K[:1].repeat(S, 0) + rng.standard_normal((S, nkv * hd)), Voh, nq, nkv, hd)
    w = w.reshape(nq, hd)
    assert np.all(w > 0) and np.allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    # huge scores do not overflow (the max is subtracted)
    Kbig = np.full((3, nkv * hd), 1e3)
    o = oracle.attention(np.full(nq * hd, 1e3), Kbig, V[:3], nq, nkv, hd)
    assert np.all(np.isfinite(o))


def test_attention_gqa_mapping():
    nq, nkv, hd, S = 4, 2, 4, 5
    rng = np.random.default_rng(1)
    K = rng.standard_normal((S, nkv * hd))
    V = np.zeros((S, nkv * hd))
    V[:, hd:] = 9.0  # only kv head 1 carries a value
    o = oracle.attention(rng.standard_normal(nq * hd), K, V, nq, nkv, hd).reshape(nq, hd)
    assert np.allclose(o[:2], 0.0) and np.allclose(o[2:], 9.0)
    # kv_group 1 is plain multi-head attention
    K2 = rng.standard_normal((S, nq * hd))
    V2 = rng.standard_normal((S, nq * hd))
    q2 = rng.standard_normal(nq * hd)
    assert np.allclose(oracle.attention(q2, K2, V2, nq, nq, hd), scipy_attention(q2, K2, V2, nq, nq, hd),
                       rtol=1e-13)


# ----------------------------------------------------------------- SiLU, argmax

def test_silu():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0)) < 1e-15
    rng = P1Rng(5)
    a = rng.vec(3072).astype(np.float64)
    b = rng.vec(3072).astype(np.float64)
    assert np.allclose(oracle.silu_mul(a, b), a * scipy_special.expit(a) * b, rtol=1e-14, atol=1e-16)


def test_argmax_planted_tie_and_nan():
    n = 151936
    x = P1Rng(77).vec(n).astype(np.float64)
    x[140011] = 9.5
    x[140012] = 9.5
    assert oracle.argmax(x) == 140011
    assert int(np.argmax(x)) == 140011  # numpy also takes the first maximum
    y = np.array([np.nan, 1.0, 3.0, np.nan, 3.0])
    assert oracle.argmax(y) == 2
    assert oracle.argmax(np.array([np.nan, np.nan])) == -1
    assert oracle.argmax(np.array([-np.inf, -np.inf])) == 0
    r = np.random.default_rng(4).standard_normal(1000)
    assert oracle.argmax(r) == int(np.argmax(r))


# ----------------------------------------------------------------- the whole step

def _rms(x, g, eps):
    return x / np.sqrt((x * x).mean() + eps) * g.astype(np.float64)


def test_step_zero_weights_is_closed_form():
    """All seven projection matrices zero: every layer is the identity, so the
    residual stays E[t] and logits = W_lm . rmsnorm(E[t]) * g_out."""
    cfg = synth.TINY
    m = synth.make_model(cfg, 0, zero_matrices=("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"))
    om = oracle.OracleModel(m, 8)
    tok = 1234
    nxt, logits = om.step(tok, 0)
    E = np_dequant_q8_0(m.lm_head, cfg.hidden)
    assert np.array_equal(om.hidden(), E[tok])
    ref = E @ _rms(E[tok], m.out_norm, cfg.rms_eps)
    assert np.allclose(logits, ref, rtol=1e-12, atol=1e-13)
    assert nxt == int(np.argmax(ref))


def test_step_attention_path_at_position_zero():
    """With only W_v and W_o non-zero, the single cached row makes attention
    return v, so each layer adds W_o W_v rmsnorm(x) to the residual."""
    cfg = synth.TINY
    m = synth.make_model(cfg, 0, zero_matrices=("wq", "wk", "w_gate", "w_up", "w_down"))
    om = oracle.OracleModel(m, 8)
    tok = 77
    om.step(tok, 0)
    x = np_dequant_q8_0(m.lm_head, cfg.hidden)[tok]
    H, qw, kvw = cfg.hidden, cfg.q_width, cfg.kv_width
    g = cfg.n_heads // cfg.n_kv_heads
    for d in m.layers:
        v = np_dequant_q8_0(d["wv"], H) @ _rms(x, d["attn_norm"], cfg.rms_eps)
        att = np.concatenate([v[(h // g) * cfg.head_dim:(h // g + 1) * cfg.head_dim] for h in range(cfg.n_heads)])
        x = x + np_dequant_q8_0(d["wo"], qw) @ att
    assert np.allclose(om.hidden(), x, rtol=1e-12, atol=1e-14)
    assert kvw == 128


def test_step_ffn_path():
    """With the attention matrices zero, each layer adds
    W_down (silu(W_gate n) * (W_up n)), n = rmsnorm(x, g_ffn)."""
    cfg = synth.TINY
    m = synth.make_model(cfg, 0, zero_matrices=("wq", "wk", "wv", "wo"))
    om = oracle.OracleModel(m, 8)
    tok = 4095
    om.step(tok, 0)
    x = np_dequant_q8_0(m.lm_head, cfg.hidden)[tok]
    for d in m.layers:
        n = _rms(x, d["ffn_norm"], cfg.rms_eps)
        gt = np_dequant_q8_0(d["w_gate"], cfg.hidden) @ n
        up = np_dequant_q8_0(d["w_up"], cfg.hidden) @ n
        x = x + np_dequant_q8_0(d["w_down"], cfg.intermediate) @ (gt * scipy_special.expit(gt) * up)
    assert np.allclose(om.hidden(), x, rtol=1e-12, atol=1e-14)


def test_step_kv_cache_rows():
    """The cached K row is the QK-normed, rotated k; with unit k-norm gains
    each head keeps norm sqrt(hd * ms/(ms+eps)) after rotation; V rows are
    the raw v projection; rows of later positions are appended, not moved."""
    cfg = synth.TINY
    m = synth.make_model(cfg, 0)
    for d in m.layers:
        d["k_norm"] = np.ones(cfg.head_dim, dtype=np.float32)
    om = oracle.OracleModel(m, 8)
    om.step(5, 0, want_logits=False)
    k0, v0 = om.kv_row(0, 0)
    om.step(6, 1, want_logits=False)
    k0b, v0b = om.kv_row(0, 0)
    assert np.array_equal(k0, k0b) and np.array_equal(v0, v0b)
    k1, _ = om.kv_row(1, 1)
    heads = k1.reshape(cfg.n_kv_heads, cfg.head_dim)
    norms = np.sqrt((heads ** 2).sum(axis=1))
    assert np.allclose(norms, math.sqrt(cfg.head_dim), rtol=1e-4)
    # V at layer 0, position 0 is W_v rmsnorm(E[5])
    E = np_dequant_q8_0(m.lm_head, cfg.hidden)
    d = m.layers[0]
    assert np.allclose(v0, np_dequant_q8_0(d["wv"], cfg.hidden) @ _rms(E[5], d["attn_norm"], cfg.rms_eps),
                       rtol=1e-12, atol=1e-14)


def test_prefill_is_repeated_steps_and_deterministic():
    cfg = synth.TINY
    m = synth.make_model(cfg, 0)
    ids = synth.token_ids(1000, 0, 6, cfg.vocab)
    a = oracle.OracleModel(m, 16)
    n1, l1 = a.prefill(ids)
    b = oracle.OracleModel(m, 16)
    for i, t in enumerate(ids):
        n2, l2 = b.step(int(t), i)
    assert n1 == n2 and np.array_equal(l1, l2)
    assert a.next_pos == len(ids)
    # re-running the last position reproduces it exactly
    n3, l3 = b.step(int(ids[-1]), len(ids) - 1)
    assert n3 == n2 and np.array_equal(l3, l2)


def test_step_rejects_bad_positions():
    m = synth.make_model(synth.TINY, 0)
    om = oracle.OracleModel(m, 4)
    with pytest.raises(ValueError):
        om.step(1, 1)  # skips position 0
    with pytest.raises(ValueError):
        om.step(synth.TINY.vocab, 0)


def _scaled_q8_scales(w: np.ndarray, factor: float) -> np.ndarray:
    """Q8_0 bytes with every block's f16 scale multiplied by `factor` (a power
    of two that keeps the scales normal, so the product is exact in f16)."""
    out = w.copy()
    blocks = out.reshape(-1, 34)
    s = blocks[:, :2].copy().view(np.float16).astype(np.float64)
    t = (s * factor).astype(np.float16)
    assert np.array_equal(t.astype(np.float64), s * factor)
    blocks[:, :2] = t.view(np.uint8).reshape(-1, 2)
    return out


def _qk_logits(m, ids):
    om = oracle.OracleModel(m, 16)
    _, logits = om.prefill(ids)
    return logits


def test_qk_norm_removes_the_scale_of_q_and_k():
    """Per-head RMSNorm of q and of k ("Eight kernels", rms_norm_row, applied
    after the projections): with eps = 0 it is invariant to a positive scale
    of its input, so multiplying every Q8_0 scale of W_q (then of W_k) by 4
    leaves the logits unchanged, while the same change to W_v (which is not
    normed) changes them.  Fails if the oracle drops the q side of the norm."""
    cfg = dataclasses.replace(synth.TINY, rms_eps=0.0)
    m = synth.make_model(cfg, 3)
    ids = synth.token_ids(1000, 5, 6, cfg.vocab)
    base = _qk_logits(m, ids)
    scale = float(np.abs(base).max())
    for name in ("wq", "wk"):
        layers = [dict(d) for d in m.layers]
        for d in layers:
            d[name] = _scaled_q8_scales(d[name], 4.0)
        got = _qk_logits(dataclasses.replace(m, layers=layers), ids)
        assert np.max(np.abs(got - base)) <= 1e-12 * scale, name
    layers = [dict(d) for d in m.layers]
    for d in layers:
        d["wv"] = _scaled_q8_scales(d["wv"], 4.0)
    assert np.max(np.abs(_qk_logits(dataclasses.replace(m, layers=layers), ids) - base)) > 1e-3 * scale


def test_qk_norm_gains_act_on_their_own_side():
    """A constant gain c on q's norm scales every attention score by c, and so
    does the same gain on k's norm: the two models give the same logits (to
    rounding), and both differ from c = 1.  Fails if the oracle applied the
    k-norm gain to q (then the first model scales by 1 and the second by c^2)
    or skipped the q-side norm."""
    cfg = synth.TINY
    m = synth.make_model(cfg, 4)
    ids = synth.token_ids(1000, 6, 6, cfg.vocab)

    def with_gains(gq, gk):
        layers = [dict(d) for d in m.layers]
        for d in layers:
            d["q_norm"] = np.full(cfg.head_dim, gq, dtype=np.float32)
            d["k_norm"] = np.full(cfg.head_dim, gk, dtype=np.float32)
        return _qk_logits(dataclasses.replace(m, layers=layers), ids)

    one = with_gains(1.0, 1.0)
    on_q = with_gains(4.0, 1.0)
    on_k = with_gains(1.0, 4.0)
    scale = float(np.abs(one).max())
    assert np.max(np.abs(on_q - on_k)) <= 1e-12 * scale
    assert np.max(np.abs(on_q - one)) > 1e-3 * scale
