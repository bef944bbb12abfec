"""Rung one of the correctness ladder on the GPU: every operator entry point
(the same device code the decode step runs) against the oracle, on the
pages' worked shapes and tolerances and on the real model shapes with ragged
tails.  Tolerances come from tests/golden/p1_correctness_ladder.txt."""
import math

import numpy as np
import pytest

import oracle
import synth
from tests.p1_lcg import P1Rng, random_q8_bytes
from tests.test_oracle_golden import HERE, load_kv

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = {k: float(v) for k, v in load_kv(f"{HERE}/p1_correctness_ladder.txt").items() if k.startswith("tol_")}


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import token_quantized_decode_gb300 as tqd
    return tqd.ops


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def q8_rows_on_device(ops, w_blocks: np.ndarray, rows: int, cols: int):
    row_bytes = (cols + cols // 16 + 15) // 16 * 16
    wb = dev(w_blocks.reshape(-1))
    wr = torch.zeros(rows * row_bytes, dtype=torch.uint8, device="cuda")
    ops.tqd_op_q8_0_repack(wb, rows, cols, wr)
    return wr


def gpu_q8_matvec(ops, w_blocks, rows, cols, x):
    wr = q8_rows_on_device(ops, w_blocks, rows, cols)
    xd = dev(np.asarray(x, dtype=np.float32))
    y = torch.full((rows,), float("nan"), device="cuda")
    ops.tqd_op_q8_0_matvec(wr, rows, cols, xd, y)
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


def abs_products(w_blocks, cols, x):
    from tests.test_oracle_pins import np_dequant_q8_0
    return np.abs(np_dequant_q8_0(w_blocks, cols)) @ np.abs(np.asarray(x, dtype=np.float64))


# ----------------------------------------------------------------- Q8_0 matvec

def test_q8_matvec_p1_case(ops):
    p, n = 50, 96
    w = random_q8_bytes(p, n, 7)
    x = P1Rng(42).vec(n)
    got = gpu_q8_matvec(ops, w, p, n, x)
    ref = oracle.q8_0_matvec(w, n, x.astype(np.float64))
    assert np.max(np.abs(got - ref)) < TOL["tol_q8_matvec"]


def test_q8_matvec_exact_integer_case_is_bit_exact(ops):
    rng = np.random.default_rng(5)
    rows, cols = 4099, 1024  # several row groups and a ragged tail
    quants = rng.integers(-127, 128, size=(rows, cols // 32, 32))
    exps = rng.integers(-4, 4, size=(rows, cols // 32))
    sbits = (15 + exps).astype(np.uint16) << 10
    w = np.zeros((rows, cols // 32, 34), dtype=np.uint8)
    w[:, :, 0] = sbits & 0xFF
    w[:, :, 1] = sbits >> 8
    w[:, :, 2:] = quants.astype(np.int8).view(np.uint8)
    w = w.reshape(rows, -1)
    x = rng.integers(-8, 9, size=cols).astype(np.float32)
    got = gpu_q8_matvec(ops, w, rows, cols, x)
    ref = oracle.q8_0_matvec(w, cols, x.astype(np.float64))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("rows,cols", [(4096, 1024), (1024, 2048), (6144, 1024), (1024, 3072),
                                       (1027, 1024), (77, 768), (33, 256), (5, 96)])
def test_q8_matvec_model_shapes(ops, rows, cols):
    w = synth.q8_0_matrix(11, rows + cols, rows, cols)
    x = synth.normal_f32(11, 7, cols, 0.0, 1.0)
    got = gpu_q8_matvec(ops, w, rows, cols, x)
    ref = oracle.q8_0_matvec(w, cols, x.astype(np.float64))
    bound = 2e-6 * abs_products(w, cols, x) + 1e-30
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))


def test_q8_matvec_lm_head_shape(ops):
    rows, cols = 151936, 1024
    w = synth.q8_0_matrix(0, 0, rows, cols)
    x = synth.normal_f32(3, 3, cols, 0.0, 1.0)
    got = gpu_q8_matvec(ops, w, rows, cols, x)
    ref = oracle.q8_0_matvec(w, cols, x.astype(np.float64))
    bound = 2e-6 * abs_products(w, cols, x)
    assert np.all(np.abs(got - ref) <= bound)


def test_q8_repack_layout(ops):
    rows, cols = 3, 256
    w = synth.q8_0_matrix(2, 2, rows, cols)
    wr = q8_rows_on_device(ops, w, rows, cols).cpu().numpy().reshape(rows, -1)
    blk = w.reshape(rows, cols // 32, 34)
    assert np.array_equal(wr[:, :cols].view(np.int8), blk[:, :, 2:].reshape(rows, cols).view(np.int8))
    assert np.array_equal(wr[:, cols:cols + cols // 16].reshape(rows, -1, 2), blk[:, :, 0:2])


# ----------------------------------------------------------------- bf16 matvec

@pytest.mark.parametrize("rows,cols", [(1600, 960), (960, 960), (5120, 960), (960, 2560), (7, 8)])
def test_bf16_matvec(ops, rows, cols):
    w = synth.bf16_matrix(4, rows, rows, cols)
    x = synth.normal_f32(4, 8, cols, 0.0, 1.0)
    y = torch.full((rows,), float("nan"), device="cuda")
    ops.tqd_op_bf16_matvec(dev(w.view(np.int16)), rows, cols, dev(x), y)
    got = y.cpu().numpy().astype(np.float64)
    ref = oracle.bf16_matvec(w, x.astype(np.float64))
    wf = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bound = 2e-6 * (np.abs(wf) @ np.abs(x.astype(np.float64)))
    assert np.all(np.abs(got - ref) <= bound)


# ----------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("rows,dim", [(1, 1024), (16, 128), (3, 1000), (5, 77), (1, 960)])
def test_rmsnorm(ops, rows, dim):
    rng = P1Rng(3)
    x = rng.vec(rows * dim)
    g = (rng.vec(dim) + np.float32(1.5)).astype(np.float32)
    out = torch.empty(rows * dim, device="cuda")
    ops.tqd_op_rmsnorm(dev(x), dev(g), rows, dim, 1e-6, out)
    ref = oracle.rmsnorm(x.astype(np.float64), g, 1e-6)
    assert np.max(np.abs(out.cpu().numpy() - ref)) < TOL["tol_rmsnorm"]


# ----------------------------------------------------------------- RoPE

@pytest.mark.parametrize("hd,theta,pos", [(128, 1e6, 137), (128, 1e6, 4159), (64, 1e5, 511), (64, 1e6, 0)])
def test_rope_table_and_rotation(ops, hd, theta, pos):
    max_pos = max(pos + 1, 8)
    table = torch.empty(max_pos * hd, device="cuda")
    ops.tqd_op_rope_table(theta, hd, max_pos, table)
    t = table.cpu().numpy().astype(np.float64).reshape(max_pos, hd // 2, 2)
    i = np.arange(hd // 2)
    ang = pos * np.power(np.float64(np.float32(theta)), -i / (hd // 2))
    assert np.max(np.abs(t[pos, :, 0] - np.cos(ang))) < 1e-7
    assert np.max(np.abs(t[pos, :, 1] - np.sin(ang))) < 1e-7
    heads = 4
    x = P1Rng(11).vec(heads * hd)
    xd = dev(x)
    ops.tqd_op_rope(xd, heads, hd, pos, table)
    ref = oracle.rope(x.astype(np.float64), heads, hd, pos, float(np.float32(theta)))
    assert np.max(np.abs(xd.cpu().numpy() - ref)) < TOL["tol_rope"]


# ----------------------------------------------------------------- attention

def gpu_attention(ops, q, K, V, nq, nkv, hd, n_chunks):
    S = K.shape[0]
    nbytes = ops.tqd_attention_scratch_bytes(nq, nkv, hd, n_chunks)
    scratch = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.full((nq * hd,), float("nan"), device="cuda")
    qd, Kd, Vd = dev(q), dev(K), dev(V)
    ops.tqd_op_attention(qd, Kd, Vd, S, nq, nkv, hd, n_chunks, out, scratch)
    torch.cuda.synchronize()
    res1 = out.cpu().numpy()
    # the scratch is left ready for reuse: a second call agrees exactly
    out.fill_(float("nan"))
    ops.tqd_op_attention(qd, Kd, Vd, S, nq, nkv, hd, n_chunks, out, scratch)
    res2 = out.cpu().numpy()
    assert np.array_equal(res1, res2)
    return res1


@pytest.mark.parametrize("nq,nkv,hd,S,chunks", [
    (4, 2, 64, 9, 1), (4, 2, 128, 9, 3), (4, 2, 64, 9, 64), (16, 8, 128, 575, 19),
    (16, 8, 128, 4160, 19), (15, 5, 64, 321, 13), (8, 8, 64, 33, 4), (8, 1, 128, 100, 7), (4, 2, 128, 1, 5)])
def test_attention(ops, nq, nkv, hd, S, chunks):
    rng = P1Rng(23)
    q = rng.vec(nq * hd) if S < 1000 else synth.uniform_f32(23, 1, nq * hd)
    K = (rng.vec(S * nkv * hd) if S < 1000 else synth.uniform_f32(23, 2, S * nkv * hd)).reshape(S, nkv * hd)
    V = (rng.vec(S * nkv * hd) if S < 1000 else synth.uniform_f32(23, 3, S * nkv * hd)).reshape(S, nkv * hd)
    got = gpu_attention(ops, q, K, V, nq, nkv, hd, chunks)
    ref = oracle.attention(q.astype(np.float64), K.astype(np.float64), V.astype(np.float64), nq, nkv, hd)
    assert np.max(np.abs(got - ref)) < TOL["tol_attention"]


def test_attention_softmax_rows_sum_to_one(ops):
    nq, nkv, hd, S = 4, 2, 64, 64
    q = synth.uniform_f32(5, 1, nq * hd, -3, 3)
    K = synth.uniform_f32(5, 2, S * nkv * hd, -3, 3).reshape(S, nkv * hd)
    V = np.tile(np.eye(hd, dtype=np.float32), (1, nkv))  # one-hot rows expose the weights
    w = gpu_attention(ops, q, K, V, nq, nkv, hd, 5).reshape(nq, hd)
    assert np.all(w >= 0) and np.allclose(w.sum(axis=1), 1.0, atol=1e-5)


# ----------------------------------------------------------------- SiLU, argmax

@pytest.mark.parametrize("n", [3072, 1000003])
def test_silu_mul(ops, n):
    rng = P1Rng(5)
    a = rng.vec(n) if n < 10000 else synth.uniform_f32(5, 1, n, -20, 20)
    b = rng.vec(n) if n < 10000 else synth.uniform_f32(5, 2, n)
    out = torch.empty(n, device="cuda")
    ops.tqd_op_silu_mul(dev(a), dev(b), n, out)
    ref = oracle.silu_mul(a.astype(np.float64), b.astype(np.float64))
    assert np.max(np.abs(out.cpu().numpy() - ref)) < TOL["tol_silu"]


def gpu_argmax(ops, x):
    scratch = torch.zeros(ops.tqd_argmax_scratch_bytes(), dtype=torch.uint8, device="cuda")
    out = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    ops.tqd_op_argmax(dev(np.asarray(x, dtype=np.float32)), len(x), out, scratch)
    return int(out.item())


def test_argmax_planted_tie(ops):
    n = 151936
    x = P1Rng(77).vec(n)
    x[140011] = 9.5
    x[140012] = 9.5
    assert gpu_argmax(ops, x) == 140011 == oracle.argmax(x.astype(np.float64))


def test_argmax_nan_and_edges(ops):
    assert gpu_argmax(ops, [float("nan"), 1.0, 3.0, float("nan"), 3.0]) == 2
    assert gpu_argmax(ops, [float("nan")] * 1000) == -1
    assert gpu_argmax(ops, [5.0]) == 0
    assert gpu_argmax(ops, [-math.inf, -math.inf]) == 0
    x = synth.uniform_f32(9, 9, 300001)
    x[[5, 299999, 123456]] = 2.0  # equal maxima far apart
    assert gpu_argmax(ops, x) == 5


def test_bounded_waits_report_a_timeout_and_the_context_survives(ops):
    """Failure detection without a fault: a wait on an mbarrier nothing arrives
    at and a wait on a counter nothing increments each give up after their
    limit, set their error bits, and the host reads TQD_ERR_DEVICE_TIMEOUT;
    the device then runs another operator normally."""
    import time
    import token_quantized_decode_gb300 as tqd
    t0 = time.perf_counter()
    status, bits = ops.tqd_op_wait_selftest()
    elapsed = time.perf_counter() - t0
    assert tqd.tqd_status_name(status) == "TQD_ERR_DEVICE_TIMEOUT"
    assert bits == 3  # counter wait (1) and mbarrier wait (2)
    assert 1.5 < elapsed < 30.0
    g = torch.randn(1000, device="cuda")
    u = torch.randn(1000, device="cuda")
    out = torch.empty(1000, device="cuda")
    ops.tqd_op_silu_mul(g, u, 1000, out)
    torch.cuda.synchronize()
    ref = (g / (1 + torch.exp(-g))) * u
    assert torch.allclose(out, ref, rtol=1e-5, atol=1e-6)
