"""Whole decode steps on the GPU against the oracle (rungs two and three of
the correctness ladder, restated for synthetic models): teacher-forced logit
parity at every step, token ids equal wherever the oracle's top-2 logit gap
exceeds 1e-2, the KV hand-over path, the chained generate path, refusals,
and the full-size workloads."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LOGIT_RTOL = 2e-3   # max |dlogit| <= 2e-3 * max |oracle logit|
TOP2_GAP = 1e-2     # token ids must agree when the oracle's top-2 gap exceeds this


@pytest.fixture(scope="module")
def tqd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import token_quantized_decode_gb300 as t
    return t


SCHEDULES = ["graph", "persistent"]


def sched(tqd, name):
    return tqd.TQD_SCHED_GRAPH if name == "graph" else tqd.TQD_SCHED_PERSISTENT


def top2_gap(logits):
    t = np.partition(logits, -2)[-2:]
    return float(t[1] - t[0])


def check_step(got_logits, got_tok, ref_logits, ref_tok, where):
    scale = float(np.max(np.abs(ref_logits)))
    err = float(np.max(np.abs(got_logits.astype(np.float64) - ref_logits)))
    assert err <= LOGIT_RTOL * scale, f"{where}: max |dlogit| {err:.3e} > {LOGIT_RTOL * scale:.3e}"
    if top2_gap(ref_logits) > TOP2_GAP:
        assert got_tok == ref_tok, f"{where}: token {got_tok} != oracle {ref_tok}"
    return err / scale


def teacher_forced(tqd, dec, om, start_pos, first_tok, n):
    """Feed the oracle's tokens to both sides for n steps; compare each."""
    tok, pos, worst = first_tok, start_pos, 0.0
    for i in range(n):
        ref_tok, ref_logits = om.step(tok, pos)
        got_tok = dec.decode_step(tok, pos)
        worst = max(worst, check_step(dec.logits(), got_tok, ref_logits, ref_tok, f"step {i} pos {pos}"))
        tok, pos = ref_tok, pos + 1
    return worst


# ----------------------------------------------------------------- tiny model

@pytest.mark.parametrize("schedule", SCHEDULES)
def test_tiny_prefill_and_teacher_forced_decode(tqd, schedule):
    wl = synth.WORKLOADS["tiny"]
    model = synth.make_model(wl.model, wl.model_seed)
    ids = synth.prompt(wl)
    max_seq = wl.prompt_len + wl.decode_steps
    om = oracle.OracleModel(model, max_seq)
    ref_tok, ref_logits = om.prefill(ids)
    dec = tqd.Decoder(model, max_seq, 1, sched(tqd, schedule))
    got_tok = dec.prefill(ids)
    check_step(dec.logits(), got_tok, ref_logits, ref_tok, "prefill")
    assert dec.next_pos() == wl.prompt_len
    teacher_forced(tqd, dec, om, wl.prompt_len, ref_tok, wl.decode_steps)
    assert dec.next_pos() == max_seq
    # the cache is full: one more step is refused, nothing changes
    with pytest.raises(tqd.TQDError) as ei:
        dec.decode_step(ref_tok, max_seq)
    assert ei.value.name == "TQD_ERR_CAPACITY"
    dec.close()


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_tiny_generate_is_device_chained_greedy(tqd, schedule):
    wl = synth.WORKLOADS["tiny"]
    cfg = wl.model
    model = synth.make_model(cfg, 3)
    ids = synth.prompt(wl)[:12]
    n = 20
    om = oracle.OracleModel(model, len(ids) + n)
    tok, _ = om.prefill(ids)
    dec = tqd.Decoder(model, len(ids) + n, 1, sched(tqd, schedule))
    assert dec.prefill(ids) == tok
    got = dec.generate(tok, n)
    pos, cur, ref = len(ids), tok, []
    gaps = []
    for _ in range(n):
        nxt, logits = om.step(cur, pos)
        ref.append(nxt)
        gaps.append(top2_gap(logits))
        cur, pos = nxt, pos + 1
    for i in range(n):
        if gaps[i] <= TOP2_GAP:
            break  # a near tie: the trajectories may legitimately part here
        assert got[i] == ref[i], f"generated id {i}: {got[i]} != {ref[i]}"
    assert dec.next_pos() == len(ids) + n
    dec.close()


def test_kv_upload_then_decode_matches_oracle(tqd):
    """Rung two: the oracle builds the KV history, the GPU decodes from it."""
    wl = synth.WORKLOADS["tiny"]
    cfg = wl.model
    model = synth.make_model(cfg, 0)
    ids = synth.prompt(wl)[:20]
    om = oracle.OracleModel(model, 32)
    om.prefill(ids[:-1])  # positions 0..18 cached
    P = len(ids) - 1
    k = np.empty((cfg.n_layers, P, cfg.kv_width), dtype=np.float32)
    v = np.empty_like(k)
    for l in range(cfg.n_layers):
        for p in range(P):
            kr, vr = om.kv_row(l, p)
            k[l, p], v[l, p] = kr, vr
    for schedule in SCHEDULES:
        dec = tqd.Decoder(model, 32, 1, sched(tqd, schedule))
        dec.kv_upload(k, v)
        assert dec.next_pos() == P
        om2 = oracle.OracleModel(model, 32)
        om2.kv_load(k, v)
        teacher_forced(tqd, dec, om2, P, int(ids[-1]), 4)
        dec.close()


def test_refusals_and_state(tqd):
    wl = synth.WORKLOADS["tiny"]
    model = synth.make_model(wl.model, 0)
    dec = tqd.Decoder(model, 8, 2)
    with pytest.raises(tqd.TQDError) as ei:
        dec.decode_step(1, 3)
    assert ei.value.name == "TQD_ERR_POS_MISMATCH"
    with pytest.raises(tqd.TQDError) as ei:
        dec.decode_step(wl.model.vocab, 0)
    assert ei.value.name == "TQD_ERR_BAD_ARG"
    with pytest.raises(tqd.TQDError) as ei:
        dec.prefill(np.arange(9))
    assert ei.value.name == "TQD_ERR_CAPACITY"
    with pytest.raises(tqd.TQDError) as ei:
        dec.decode_step(1, 0, seq=2)
    assert ei.value.name == "TQD_ERR_BAD_ARG"
    # nothing above changed the sequence; a step and a replay after reset agree bitwise
    assert dec.next_pos() == 0
    a = dec.decode_step(17, 0)
    la = dec.logits()
    dec.reset()
    b = dec.decode_step(17, 0)
    assert a == b and np.array_equal(la, dec.logits())
    # sequences are independent
    c = dec.decode_step(17, 0, seq=1)
    assert c == a and np.array_equal(la, dec.logits(seq=1))
    assert dec.phase_count == 5 * wl.model.n_layers + 2
    dec.close()
    dp = tqd.Decoder(model, 8, 1, tqd.TQD_SCHED_PERSISTENT)
    assert dp.phase_count == 4 * wl.model.n_layers + 1
    dp.close()


def test_step_bytes_match_the_shapes(tqd):
    # Qwen3-0.6B shape: 28 layers x 16,711,680 B + lm_head 165,306,368 B +
    # f32 norms 262,144 B + one embedding row 1,088 B; 229,376 KV bytes per position
    model = synth.make_model(synth.TINY, 0)
    dec = tqd.Decoder(model, 8)
    cfg = synth.TINY
    per_layer = ((cfg.q_width + 2 * cfg.kv_width) * 272 + cfg.hidden * 272 + 2 * cfg.intermediate * 272 +
                 cfg.hidden * 816 + 4 * (2 * cfg.hidden + 2 * cfg.head_dim))
    weights = cfg.n_layers * per_layer + cfg.vocab * 272 + 4 * cfg.hidden + 272
    kv = 4 * cfg.kv_width * 2 * cfg.n_layers
    assert dec.step_bytes(5) == weights + kv * 6 + kv
    dec.close()


# ----------------------------------------------------------------- full sizes

def reference_run(model, ids, max_seq, n_steps):
    """The oracle's prefill and n_steps greedy steps: [(token, pos, logits, next)]."""
    om = oracle.OracleModel(model, max_seq)
    tok, logits = om.prefill(ids)
    out = [(None, None, logits, tok)]
    pos = len(ids)
    for _ in range(n_steps):
        nxt, lg = om.step(tok, pos)
        out.append((tok, pos, lg, nxt))
        tok, pos = nxt, pos + 1
    return out


def replay(dec, ids, ref, tiles=False):
    got = dec.prefill_batch(ids) if tiles else dec.prefill(ids)
    check_step(dec.logits(), got, ref[0][2], ref[0][3], "prefill")
    for i, (tok, pos, lg, nxt) in enumerate(ref[1:]):
        got = dec.decode_step(tok, pos)
        check_step(dec.logits(), got, lg, nxt, f"step {i} pos {pos}")


@pytest.fixture(scope="module")
def qwen3_reference():
    wl = synth.WORKLOADS["qwen3_0.6b"]
    model = synth.make_model(wl.model, wl.model_seed)
    ids = synth.prompt(wl)
    return wl, model, ids, reference_run(model, ids, wl.prompt_len + 8, 8)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_qwen3_shape_full_size(tqd, qwen3_reference, schedule):
    """Qwen3-0.6B shape, 511-token prompt prefilled on the GPU, then eight
    teacher-forced decode steps, in the launch configuration the benchmark
    times."""
    wl, model, ids, ref = qwen3_reference
    dec = tqd.Decoder(model, wl.prompt_len + wl.decode_steps, 1, sched(tqd, schedule))
    replay(dec, ids, ref)
    dec.close()


def test_qwen3_shape_prefill_tiles_full_size(tqd, qwen3_reference):
    """The same 511-token prompt prefilled in tiles of 16 (31 full tiles and
    one of 15) on the one-sequence persistent model the benchmark times, then
    the eight teacher-forced decode steps over the cache the tiles wrote."""
    wl, model, ids, ref = qwen3_reference
    dec = tqd.Decoder(model, wl.prompt_len + wl.decode_steps, 1, tqd.TQD_SCHED_PERSISTENT)
    replay(dec, ids, ref, tiles=True)
    dec.close()


def test_smollm2_shape_bf16_full_size(tqd):
    wl = synth.WORKLOADS["smollm2_360m"]
    model = synth.make_model(wl.model, wl.model_seed)
    ids = synth.prompt(wl)
    ref = reference_run(model, ids, wl.prompt_len + 4, 4)
    for schedule in SCHEDULES:
        dec = tqd.Decoder(model, wl.prompt_len + wl.decode_steps, 1, sched(tqd, schedule))
        replay(dec, ids, ref)
        dec.close()


def test_qwen3_long_context_from_uploaded_kv(tqd):
    """4096 cached positions (seeded stand-in history), then decode steps
    that scan all of them through the split-K attention."""
    wl = synth.WORKLOADS["qwen3_0.6b_long"]
    cfg = wl.model
    model = synth.make_model(cfg, wl.model_seed)
    k, v = synth.kv_fill(cfg, 7, 0, wl.prompt_len, -1.0, 1.0)
    for schedule in SCHEDULES:
        om = oracle.OracleModel(model, wl.prompt_len + 5)
        om.kv_load(k, v)
        dec = tqd.Decoder(model, wl.prompt_len + 64, 1, sched(tqd, schedule))
        dec.kv_upload(k, v)
        teacher_forced(tqd, dec, om, wl.prompt_len, 12345, 4)
        dec.close()
