"""The allocation-free attention entry point, for callers that may not
allocate device memory while they run (its scratch is a static device array
inside the library).  Its results must equal those of tqd_op_attention, which
takes caller-allocated scratch, on two calls in a row.  Kept in a file of its
own that pytest collects last."""
import numpy as np
import pytest

import synth
from tests.test_oracle_golden import HERE, load_kv

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = float(load_kv(f"{HERE}/p1_correctness_ladder.txt")["tol_attention"])


def test_attention_noalloc_matches_scratch_variant_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import token_quantized_decode_gb300 as tqd
    ops = tqd.ops
    nq, nkv, hd, S, chunks = 16, 8, 128, 575, 19
    assert ops.tqd_attention_scratch_bytes(nq, nkv, hd, chunks) <= ops.tqd_op_attention_noalloc_max_scratch()
    q = torch.from_numpy(synth.uniform_f32(31, 1, nq * hd)).cuda()
    K = torch.from_numpy(synth.uniform_f32(31, 2, S * nkv * hd)).cuda()
    V = torch.from_numpy(synth.uniform_f32(31, 3, S * nkv * hd)).cuda()
    scratch = torch.zeros(ops.tqd_attention_scratch_bytes(nq, nkv, hd, chunks), dtype=torch.uint8, device="cuda")
    ref = torch.full((nq * hd,), float("nan"), device="cuda")
    ops.tqd_op_attention(q, K, V, S, nq, nkv, hd, chunks, ref, scratch)
    ref_h = ref.cpu().numpy()
    for _ in range(2):
        out = torch.full((nq * hd,), float("nan"), device="cuda")
        ops.tqd_op_attention_noalloc(q, K, V, S, nq, nkv, hd, chunks, out)
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - ref_h)) <= TOL
    # a request larger than the static array is refused, not run
    with pytest.raises(tqd.TQDError) as ei:
        ops.tqd_op_attention_noalloc(q, K, V, S, nq, nkv, hd, 1024, out)
    assert ei.value.name == "TQD_ERR_BAD_ARG"
