"""tqd_create_synthetic (the seeded synthetic model generated inside the
library, so that a C caller loads the benchmark's model with one call) and
tqd_export_weights (the weights read back in the upload format): the exported
bytes equal the Python generator's for the same seed, bit for bit, and the
model's steps match the oracle on those bytes."""
import numpy as np
import pytest

import oracle
import synth
from tests.test_gpu_decode import check_step

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BF16_SMALL = synth.ModelConfig(2, 256, 6, 2, 64, 768, 4096, False, "bf16", 1e5)


@pytest.fixture(scope="module")
def tqd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import token_quantized_decode_gb300 as t
    return t


def assert_same_weights(got, ref):
    assert np.array_equal(got["lm_head"], ref.lm_head)
    assert np.array_equal(got["out_norm"], ref.out_norm)
    for l, (g, r) in enumerate(zip(got["layers"], ref.layers)):
        assert set(g) == set(r), l
        for name in r:
            assert np.array_equal(g[name], r[name]), (l, name)


@pytest.mark.parametrize("cfg, schedule", [(synth.TINY, "persistent"), (BF16_SMALL, "graph")])
def test_synthetic_model_is_the_generator_model(tqd, cfg, schedule):
    seed = 5
    sched = tqd.TQD_SCHED_PERSISTENT if schedule == "persistent" else tqd.TQD_SCHED_GRAPH
    dec = tqd.Decoder.synthetic(cfg, seed, 32, 1, sched)
    ref = synth.make_model(cfg, seed)
    assert_same_weights(dec.export_weights(), ref)
    ids = synth.token_ids(1000, 3, 12, cfg.vocab)
    om = oracle.OracleModel(ref, 32)
    tok, lg = om.prefill(ids)
    got = dec.prefill(ids)
    check_step(dec.logits(), got, lg, tok, "prefill")
    p = len(ids)
    for i in range(3):
        ref_tok, ref_lg = om.step(tok, p)
        got = dec.decode_step(tok, p)
        check_step(dec.logits(), got, ref_lg, ref_tok, f"step {i}")
        tok, p = ref_tok, p + 1
    dec.close()


def test_synthetic_qwen3_shape_equals_the_generator(tqd):
    """The benchmark's Qwen3-0.6B-shape model (seed 0), every tensor."""
    wl = synth.WORKLOADS["qwen3_0.6b"]
    dec = tqd.Decoder.synthetic(wl.model, wl.model_seed, 8, 1, tqd.TQD_SCHED_PERSISTENT)
    got = dec.export_weights()
    dec.close()
    assert_same_weights(got, synth.make_model(wl.model, wl.model_seed))


def test_export_of_an_uploaded_model_round_trips(tqd):
    """Weights uploaded from host arrays come back byte for byte (the
    interleaved gate/up rows, the repacked Q8_0 rows)."""
    model = synth.make_model(synth.TINY, 9)
    dec = tqd.Decoder(model, 8, 2)
    assert_same_weights(dec.export_weights(), model)
    dec.close()


@pytest.mark.parametrize("schedule", ["persistent", "graph"])
def test_c_client_generates_the_oracle_tokens(tqd, schedule):
    """tests/c/tqd_client.c, a C program using the C ABI alone
    (tqd_create_synthetic, tqd_prefill, tqd_generate), prints the oracle's
    greedy tokens for the seeded tiny model.  A token may differ only where
    the oracle's two candidates lie within the decode tests' top-2 gap (then the
    sequences part and the comparison stops)."""
    import subprocess
    import tempfile
    from tests.test_abi import _build_client
    from tests.test_gpu_decode import TOP2_GAP
    cfg, seed, steps = synth.TINY, 5, 8
    ids = synth.token_ids(1000, 3, 12, cfg.vocab)
    sched = tqd.TQD_SCHED_PERSISTENT if schedule == "persistent" else tqd.TQD_SCHED_GRAPH
    shape = (cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.intermediate, cfg.vocab,
             int(cfg.qk_norm), 0 if cfg.weight_type == "q8_0" else 1)
    with tempfile.TemporaryDirectory() as d:
        exe = _build_client(d)
        args = [exe, str(seed), str(steps), str(sched), *map(str, shape), repr(cfg.rope_theta), repr(cfg.rms_eps),
                *(str(int(t)) for t in ids)]
        r = subprocess.run(args, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    got = [int(x) for x in r.stdout.split()]
    assert len(got) == steps + 1
    om = oracle.OracleModel(synth.make_model(cfg, seed), len(ids) + steps + 1)
    tok, lg = om.prefill(ids)
    p = len(ids)
    for i in range(steps + 1):
        if got[i] != tok:
            assert lg[tok] - lg[got[i]] <= TOP2_GAP, (i, got[i], tok)
            break
        if i < steps:
            tok, lg = om.step(tok, p)
            p += 1
