"""An f16 KV cache (TQD_KV_F16: every cached K and V element rounded to the
nearest binary16 as it is appended or uploaded) in the batched step, the
prefill tiles and both batch-1 schedules, against the oracle with the same
rounding step, at the whole step's tolerance (the device rounds its f32 rows, the oracle its f64 rows, so
an element can land one f16 step apart)."""
import numpy as np
import pytest

import oracle
import synth
from tests.test_gpu_decode import check_step

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tqd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import token_quantized_decode_gb300 as t
    return t


def test_kv16_prefill_tiles_then_batched_steps(tqd):
    """Four sequences prefilled in tiles (9, 16, 23 and 40 positions), then
    three teacher-forced batched steps at their different positions."""
    cfg = synth.TINY
    model = synth.make_model(cfg, 21)
    lens = [9, 16, 23, 40]
    n, max_seq = len(lens), 48
    dec = tqd.Decoder(model, max_seq, n, kv_type=tqd.TQD_KV_F16)
    oms, toks, pos = [], [], []
    for b, P in enumerate(lens):
        ids = synth.token_ids(1000, 60 + b, P, cfg.vocab)
        om = oracle.OracleModel(model, max_seq, kv_f16=True)
        tok, lg = om.prefill(ids)
        got = dec.prefill_batch(ids, seq=b)
        check_step(dec.logits(seq=b), got, lg, tok, f"prefill seq {b}")
        oms.append(om)
        toks.append(tok)
        pos.append(P)
    for i in range(3):
        refs = [oms[b].step(toks[b], pos[b]) for b in range(n)]
        got = dec.decode_step_batch(np.array(toks), np.array(pos))
        for b in range(n):
            check_step(dec.logits(seq=b), int(got[b]), refs[b][1], refs[b][0], f"step {i} seq {b}")
        toks = [r[0] for r in refs]
        pos = [p + 1 for p in pos]
    dec.close()


def test_kv16_one_sequence_model(tqd):
    """max_batch 1: the batched entry points run an f16 cache for a single
    sequence (prefill tiles, batched steps of one, a seeded draw)."""
    cfg = synth.ModelConfig(2, 256, 6, 2, 64, 768, 4096, False, "bf16", 1e5)
    model = synth.make_model(cfg, 22)
    ids = synth.token_ids(1000, 70, 37, cfg.vocab)
    om = oracle.OracleModel(model, 48, kv_f16=True)
    tok, lg = om.prefill(ids)
    dec = tqd.Decoder(model, 48, 1, kv_type=tqd.TQD_KV_F16)
    got = dec.prefill_batch(ids)
    check_step(dec.logits(), got, lg, tok, "prefill")
    p = len(ids)
    for i in range(3):
        ref_tok, ref_lg = om.step(tok, p)
        got = dec.decode_step_batch(np.array([tok]), np.array([p]))
        check_step(dec.logits(), int(got[0]), ref_lg, ref_tok, f"step {i}")
        tok, p = ref_tok, p + 1
    assert 0 <= dec.sample(tqd.sampling(temperature=0.9, top_k=20, seed=3)) < cfg.vocab
    dec.close()


def test_kv16_uploaded_history(tqd):
    """Seeded f32 histories uploaded (rounded to f16 on the way) to three
    sequences, then two batched steps."""
    cfg = synth.TINY
    model = synth.make_model(cfg, 23)
    n, P = 3, 30
    dec = tqd.Decoder(model, P + 4, n, kv_type=tqd.TQD_KV_F16)
    oms, toks = [], []
    for b in range(n):
        k, v = synth.kv_fill(cfg, 80 + b, b, P)
        dec.kv_upload(k, v, seq=b)
        om = oracle.OracleModel(model, P + 4, kv_f16=True)
        om.kv_load(k, v)
        oms.append(om)
        toks.append(int(synth.token_ids(1000, 90 + b, 1, cfg.vocab)[0]))
    pos = [P] * n
    for i in range(2):
        refs = [oms[b].step(toks[b], pos[b]) for b in range(n)]
        got = dec.decode_step_batch(np.array(toks), np.array(pos))
        for b in range(n):
            check_step(dec.logits(seq=b), int(got[b]), refs[b][1], refs[b][0], f"step {i} seq {b}")
        toks = [r[0] for r in refs]
        pos = [p + 1 for p in pos]
    dec.close()


def test_kv16_shape_outside_the_batched_kernels(tqd):
    """8 q heads per kv head: the batched kernels refuse the shape, the graph
    schedule runs it on an f16 cache (against the oracle's)."""
    wide = synth.ModelConfig(1, 256, 8, 1, 64, 512, 4096, True, "q8_0", 1e6)
    model = synth.make_model(wide, 0)
    dec = tqd.Decoder(model, 16, 1, tqd.TQD_SCHED_GRAPH, kv_type=tqd.TQD_KV_F16)
    with pytest.raises(tqd.TQDError) as ei:
        dec.prefill_batch([1, 2, 3])
    assert ei.value.name == "TQD_ERR_UNSUPPORTED_CONFIG"
    om = oracle.OracleModel(model, 16, kv_f16=True)
    tok, lg = om.prefill([1, 2, 3])
    got = dec.prefill([1, 2, 3])
    check_step(dec.logits(), got, lg, tok, "prefill")
    dec.close()


@pytest.mark.parametrize("schedule", ["graph", "persistent"])
def test_kv16_batch1_schedules(tqd, schedule):
    """The batch-1 schedules on an f16 cache: a stepwise prefill of 19
    positions, four teacher-forced steps, then a chained generate whose
    steps are replayed one by one on the oracle's f16 cache."""
    cfg = synth.TINY
    model = synth.make_model(cfg, 24)
    ids = synth.token_ids(1000, 71, 19, cfg.vocab)
    sched = tqd.TQD_SCHED_GRAPH if schedule == "graph" else tqd.TQD_SCHED_PERSISTENT
    om = oracle.OracleModel(model, 40, kv_f16=True)
    tok, lg = om.prefill(ids)
    dec = tqd.Decoder(model, 40, 1, sched, kv_type=tqd.TQD_KV_F16)
    got = dec.prefill(ids)
    check_step(dec.logits(), got, lg, tok, "prefill")
    p = len(ids)
    for i in range(4):
        ref_tok, ref_lg = om.step(tok, p)
        got = dec.decode_step(tok, p)
        check_step(dec.logits(), got, ref_lg, ref_tok, f"step {i}")
        tok, p = ref_tok, p + 1
    ids_gen = dec.generate(tok, 6)
    for i in range(6):  # the oracle follows the device's own chain
        ref_tok, ref_lg = om.step(tok, p + i)
        top2 = np.sort(ref_lg)[-2:]
        if top2[1] - top2[0] > 1e-2:
            assert int(ids_gen[i]) == ref_tok, f"generated step {i}"
        tok = int(ids_gen[i])
    dec.close()


@pytest.mark.parametrize("schedule", ["graph", "persistent"])
def test_kv16_qwen3_long_history_batch1(tqd, schedule):
    """Qwen3-0.6B shape with a 4096-position history uploaded into an f16
    cache (rounded on the way, as the oracle rounds its copy), then three
    teacher-forced steps at positions 4096..4098 on a batch-1 schedule."""
    wl = synth.WORKLOADS["qwen3_0.6b_long"]
    cfg = wl.model
    model = synth.make_model(cfg, wl.model_seed)
    P = 4096
    k, v = synth.kv_fill(cfg, 7, 0, P)
    sched = tqd.TQD_SCHED_GRAPH if schedule == "graph" else tqd.TQD_SCHED_PERSISTENT
    dec = tqd.Decoder(model, P + 4, 1, sched, kv_type=tqd.TQD_KV_F16)
    dec.kv_upload(k, v)
    om = oracle.OracleModel(model, P + 4, kv_f16=True)
    om.kv_load(k, v)
    del k, v
    tok = int(synth.prompt(wl)[-1])
    for i in range(3):
        ref_tok, ref_lg = om.step(tok, P + i)
        got = dec.decode_step(tok, P + i)
        check_step(dec.logits(), got, ref_lg, ref_tok, f"step {i}")
        tok = ref_tok
    dec.close()


def test_kv16_qwen3_shape_sixteen_sequences(tqd):
    """Qwen3-0.6B shape, 16 sequences with uploaded 1024-position histories,
    two teacher-forced batched steps; sequences 0 and 11 against the oracle."""
    wl = synth.WORKLOADS["qwen3_0.6b_batch16"]
    cfg = wl.model
    model = synth.make_model(cfg, wl.model_seed)
    n, P = 16, 1024
    dec = tqd.Decoder(model, P + 4, n, kv_type=tqd.TQD_KV_F16)
    toks, oms = [], {}
    for b in range(n):
        k, v = synth.kv_fill(cfg, 40 + b, b, P)
        dec.kv_upload(k, v, seq=b)
        if b in (0, 11):
            om = oracle.OracleModel(model, P + 4, kv_f16=True)
            om.kv_load(k, v)
            oms[b] = om
        toks.append(int(synth.token_ids(1000, b, 1, cfg.vocab)[0]))
    pos = [P] * n
    for i in range(2):
        refs = {b: oms[b].step(toks[b], pos[b]) for b in oms}
        got = dec.decode_step_batch(np.array(toks), np.array(pos))
        for b in oms:
            check_step(dec.logits(seq=b), int(got[b]), refs[b][1], refs[b][0], f"step {i} seq {b}")
        toks = [refs[b][0] if b in refs else int(got[b]) for b in range(n)]
        pos = [p + 1 for p in pos]
    dec.close()
