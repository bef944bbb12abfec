"""The batched decode step (several sequences per step, tensor-core
contractions for the projections) against the oracle, one oracle model per
sequence, teacher-forced."""
import numpy as np
import pytest

import oracle
import synth
from tests.test_gpu_decode import check_step, top2_gap, TOP2_GAP

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tqd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import token_quantized_decode_gb300 as t
    return t


def batched_vs_oracle(tqd, cfg, n_seq, prompt_len, steps, max_seq, seed=0, kv_history=0):
    """Prefill (or upload a seeded history for) n_seq sequences, then run
    `steps` teacher-forced batched steps; compare every sequence's logits."""
    model = synth.make_model(cfg, seed)
    dec = tqd.Decoder(model, max_seq, n_seq)
    oms, toks, pos = [], [], []
    for b in range(n_seq):
        om = oracle.OracleModel(model, max_seq)
        if kv_history:
            k, v = synth.kv_fill(cfg, 40 + b, b, kv_history)
            om.kv_load(k, v)
            dec.kv_upload(k, v, seq=b)
            tok = int(synth.token_ids(1000, b, 1, cfg.vocab)[0])
            p = kv_history
        else:
            ids = synth.token_ids(1000, b, prompt_len, cfg.vocab)
            tok, _ = om.prefill(ids)
            assert dec.prefill(ids, seq=b) == tok
            p = prompt_len
        oms.append(om)
        toks.append(tok)
        pos.append(p)
    worst = 0.0
    for i in range(steps):
        refs = [oms[b].step(toks[b], pos[b]) for b in range(n_seq)]
        got = dec.decode_step_batch(np.array(toks), np.array(pos))
        for b in range(n_seq):
            worst = max(worst, check_step(dec.logits(seq=b), int(got[b]), refs[b][1], refs[b][0],
                                          f"step {i} seq {b}"))
        toks = [r[0] for r in refs]
        pos = [p + 1 for p in pos]
    assert all(dec.next_pos(seq=b) == pos[b] for b in range(n_seq))
    dec.close()
    return worst


def test_batch_tiny_q8(tqd):
    w = batched_vs_oracle(tqd, synth.TINY, 4, 12, 4, 24)
    assert w < 1e-4  # f32-level: the three-part bf16 split keeps the contraction exact


def test_batch_tiny_bf16(tqd):
    cfg = synth.ModelConfig(2, 256, 6, 2, 64, 768, 4096, False, "bf16", 1e5)
    w = batched_vs_oracle(tqd, cfg, 3, 10, 3, 20)
    assert w < 1e-4


def test_batch_odd_shape(tqd):
    """Hidden 320 (ten 32-wide blocks: uneven cluster K splits, a half last pass
    of the lm_head) and vocabulary 4000 (a last lm_head tile of 32 rows,
    zero-padded in the tile-pass copy)."""
    cfg = synth.ModelConfig(2, 320, 4, 2, 64, 640, 4000, True, "q8_0", 1e6)
    w = batched_vs_oracle(tqd, cfg, 6, 9, 3, 16)
    assert w < 1e-4


def test_batch_sixteen_tiny_sequences(tqd):
    assert batched_vs_oracle(tqd, synth.TINY, 16, 6, 2, 12) < 1e-4


def test_batch_ragged_positions(tqd):
    """Sequences at different positions in one step (histories of 1 to 23
    rows): each sequence's attention split and the O projection's merge of its
    chunks follow its own length; three teacher-forced steps vs the oracle."""
    cfg = synth.TINY
    model = synth.make_model(cfg, 2)
    lens = [1, 4, 9, 16, 23]
    n, steps, max_seq = len(lens), 3, 32
    dec = tqd.Decoder(model, max_seq, n)
    oms, toks, pos = [], [], []
    for b, P in enumerate(lens):
        ids = synth.token_ids(1000, 20 + b, P, cfg.vocab)
        om = oracle.OracleModel(model, max_seq)
        tok, _ = om.prefill(ids)
        assert dec.prefill(ids, seq=b) == tok
        oms.append(om)
        toks.append(tok)
        pos.append(P)
    worst = 0.0
    for i in range(steps):
        refs = [oms[b].step(toks[b], pos[b]) for b in range(n)]
        got = dec.decode_step_batch(np.array(toks), np.array(pos))
        for b in range(n):
            worst = max(worst, check_step(dec.logits(seq=b), int(got[b]), refs[b][1], refs[b][0],
                                          f"step {i} seq {b} pos {pos[b]}"))
        toks = [r[0] for r in refs]
        pos = [p + 1 for p in pos]
    assert worst < 1e-4
    dec.close()


def test_batch_matches_single_sequence_path(tqd):
    cfg = synth.TINY
    model = synth.make_model(cfg, 5)
    n = 5
    single = tqd.Decoder(model, 16, 1)
    batch = tqd.Decoder(model, 16, n)
    prompts = [synth.token_ids(1000, b, 7, cfg.vocab) for b in range(n)]
    firsts = [batch.prefill(p, seq=b) for b, p in enumerate(prompts)]
    got = batch.decode_step_batch(np.array(firsts), np.full(n, 7))
    for b in range(n):
        single.reset()
        assert single.prefill(prompts[b]) == firsts[b]
        nxt = single.decode_step(firsts[b], 7)
        ref = single.logits()
        lb = batch.logits(seq=b)
        assert np.max(np.abs(lb - ref)) <= 1e-5 * np.max(np.abs(ref))
        assert nxt == got[b]
    single.close()
    batch.close()


def test_batch_generate_chained(tqd):
    cfg = synth.TINY
    model = synth.make_model(cfg, 3)
    n, P, steps = 4, 9, 6
    dec = tqd.Decoder(model, P + steps + 1, n)
    firsts, refs = [], []
    for b in range(n):
        ids = synth.token_ids(1000, b, P, cfg.vocab)
        om = oracle.OracleModel(model, P + steps + 1)
        tok, _ = om.prefill(ids)
        firsts.append(dec.prefill(ids, seq=b))
        seq, gaps, cur = [], [], tok
        for i in range(steps):
            cur, lg = om.step(cur, P + i)
            seq.append(cur)
            gaps.append(top2_gap(lg))
        refs.append((seq, gaps))
    ids = dec.generate_batch(np.array(firsts), steps)
    assert ids.shape == (steps, n)
    for b in range(n):
        seq, gaps = refs[b]
        for i in range(steps):
            if gaps[i] <= TOP2_GAP:
                break
            assert ids[i, b] == seq[i]
    dec.close()


def test_batch_refusals(tqd):
    model = synth.make_model(synth.TINY, 0)
    one = tqd.Decoder(model, 8, 1)
    with pytest.raises(tqd.TQDError) as ei:
        one.decode_step_batch([1], [0])
    assert ei.value.name == "TQD_ERR_UNSUPPORTED_CONFIG"
    one.close()
    dec = tqd.Decoder(model, 8, 2)
    with pytest.raises(tqd.TQDError) as ei:
        dec.decode_step_batch([1, 2, 3], [0, 0, 0])
    assert ei.value.name == "TQD_ERR_BAD_ARG"
    with pytest.raises(tqd.TQDError) as ei:
        dec.decode_step_batch([1, 2], [0, 1])
    assert ei.value.name == "TQD_ERR_POS_MISMATCH"
    dec.close()


def test_batch_qwen3_shape_sixteen_sequences(tqd):
    """Qwen3-0.6B shape, 16 sequences with seeded 1024-position histories,
    three batched steps; every sequence against the oracle.  The device runs
    its own chain (each step's argmax is the next input) and records every
    step's logits; then one oracle at a time takes a sequence's history and
    the same inputs, so both sides see identical tokens at every step: the
    logits must agree at every step, the tokens wherever the oracle's top-2
    gap exceeds 1e-2."""
    wl = synth.WORKLOADS["qwen3_0.6b_batch16"]
    cfg = wl.model
    model = synth.make_model(cfg, wl.model_seed)
    n, P, steps = 16, 1024, 3
    dec = tqd.Decoder(model, P + 4, n)
    toks = []
    for b in range(n):
        k, v = synth.kv_fill(cfg, 40 + b, b, P)
        dec.kv_upload(k, v, seq=b)
        toks.append(int(synth.token_ids(1000, b, 1, cfg.vocab)[0]))
    inputs, outs, logits = [], [], []
    for i in range(steps):
        got = dec.decode_step_batch(np.array(toks), np.full(n, P + i))
        inputs.append(list(toks))
        outs.append([int(t) for t in got])
        logits.append([dec.logits(seq=b) for b in range(n)])
        toks = outs[-1]
    dec.close()
    for b in range(n):
        k, v = synth.kv_fill(cfg, 40 + b, b, P)
        om = oracle.OracleModel(model, P + 4)
        om.kv_load(k, v)
        del k, v
        for i in range(steps):
            ref_tok, ref_lg = om.step(inputs[i][b], P + i)
            check_step(logits[i][b], outs[i][b], ref_lg, ref_tok, f"step {i} seq {b}")
        del om


def test_batch_beyond_sixteen_sequences(tqd):
    """32 sequences at ragged positions (prompts of 3..34 positions prefilled
    in tiles), then three teacher-forced batched steps of all 32 (two groups
    of 16, each one sweep of the weights) and two of the first 20 (a group of
    16 and one of 4): every sequence against the oracle at every step; then a
    chained generate of the 32 replayed against the oracle."""
    cfg = synth.TINY
    model = synth.make_model(cfg, 31)
    n, max_seq = 32, 48
    dec = tqd.Decoder(model, max_seq, n)
    oms, toks, pos = [], [], []
    for b in range(n):
        P = 3 + b
        ids = synth.token_ids(1000, 200 + b, P, cfg.vocab)
        om = oracle.OracleModel(model, max_seq)
        tok, lg = om.prefill(ids)
        got = dec.prefill_batch(ids, seq=b)
        check_step(dec.logits(seq=b), got, lg, tok, f"prefill seq {b}")
        oms.append(om)
        toks.append(tok)
        pos.append(P)
    for width, steps in ((32, 3), (20, 2)):
        for i in range(steps):
            refs = [oms[b].step(toks[b], pos[b]) for b in range(width)]
            got = dec.decode_step_batch(np.array(toks[:width]), np.array(pos[:width]))
            for b in range(width):
                check_step(dec.logits(seq=b), int(got[b]), refs[b][1], refs[b][0], f"{width}-wide step {i} seq {b}")
                toks[b] = refs[b][0]
                pos[b] += 1
    dec.close()
    # chained: 32 sequences, four device-chained steps, the oracle following
    # each sequence's own chain
    dec = tqd.Decoder(model, max_seq, n)
    firsts, oms = [], []
    for b in range(n):
        ids = synth.token_ids(1000, 300 + b, 5 + b % 7, cfg.vocab)
        firsts.append(dec.prefill_batch(ids, seq=b))
        om = oracle.OracleModel(model, max_seq)
        om.prefill(ids)
        oms.append((om, len(ids)))
    got = dec.generate_batch(np.array(firsts), 4)
    for b in range(n):
        om, P = oms[b]
        tok = firsts[b]
        for i in range(4):
            ref_tok, ref_lg = om.step(tok, P + i)
            top2 = np.sort(ref_lg)[-2:]
            if top2[1] - top2[0] > 1e-2:
                assert int(got[i, b]) == ref_tok, f"chained step {i} seq {b}"
            tok = int(got[i, b])
    dec.close()
