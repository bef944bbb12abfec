"""The allocation-free attention entry point, for callers that may not
allocate device memory while they run (its scratch is a static device array
inside the library).  Its results must equal those of tqd_op_attention, which
takes caller-allocated scratch, on consecutive calls, and the oracle's within
the attention tolerance.  Between two calls of one shape, a call of another
shape leaves different bytes where the first shape keeps its arrival
counters, so the per-call clearing of those counters is exercised; one shape
fills the static array to within a few hundred bytes of its size.  Kept in a
file of its own that pytest collects last."""
import numpy as np
import pytest

import oracle
import synth
from tests.test_oracle_golden import HERE, load_kv

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = float(load_kv(f"{HERE}/p1_correctness_ladder.txt")["tol_attention"])

# (n_heads, n_kv, head_dim, S, n_chunks)
SHAPES = [(16, 8, 128, 575, 19), (4, 2, 64, 200, 3), (16, 8, 128, 575, 19), (16, 8, 128, 575, 126)]


def inputs(nq, nkv, hd, S, seed):
    q = synth.uniform_f32(seed, 1, nq * hd)
    K = synth.uniform_f32(seed, 2, S * nkv * hd)
    V = synth.uniform_f32(seed, 3, S * nkv * hd)
    return q, K, V


def test_attention_noalloc_matches_scratch_variant_and_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import token_quantized_decode_gb300 as tqd
    ops = tqd.ops
    cap = ops.tqd_op_attention_noalloc_max_scratch()
    assert cap - 512 <= ops.tqd_attention_scratch_bytes(16, 8, 128, 126) <= cap
    for i, (nq, nkv, hd, S, chunks) in enumerate(SHAPES):
        assert ops.tqd_attention_scratch_bytes(nq, nkv, hd, chunks) <= cap
        qh, Kh, Vh = inputs(nq, nkv, hd, S, 31 + (i % 2))
        q, K, V = (torch.from_numpy(a).cuda() for a in (qh, Kh, Vh))
        scratch = torch.zeros(ops.tqd_attention_scratch_bytes(nq, nkv, hd, chunks), dtype=torch.uint8,
                              device="cuda")
        ref = torch.full((nq * hd,), float("nan"), device="cuda")
        ops.tqd_op_attention(q, K, V, S, nq, nkv, hd, chunks, ref, scratch)
        ref_h = ref.cpu().numpy()
        want = oracle.attention(qh.astype(np.float64), Kh.reshape(S, nkv * hd).astype(np.float64),
                                Vh.reshape(S, nkv * hd).astype(np.float64), nq, nkv, hd)
        for _ in range(2):
            out = torch.full((nq * hd,), float("nan"), device="cuda")
            ops.tqd_op_attention_noalloc(q, K, V, S, nq, nkv, hd, chunks, out)
            got = out.cpu().numpy()
            assert np.all(np.isfinite(got)), SHAPES[i]
            assert np.max(np.abs(got - ref_h)) <= TOL, SHAPES[i]
            assert np.max(np.abs(got - want)) <= TOL, SHAPES[i]
    # a request larger than the static array is refused, not run
    with pytest.raises(tqd.TQDError) as ei:
        ops.tqd_op_attention_noalloc(q, K, V, S, nq, nkv, hd, 127, out)
    assert ei.value.name == "TQD_ERR_BAD_ARG"
