"""Prefill in tiles of up to 16 positions (tqd_prefill_batch: one batched
step per tile, the tile's slots attending to each other's rows) against the
oracle's prefill, which runs the decode step over the prompt position by
position; every test continues with decode steps that attend to every cached
row the tiles wrote."""
import numpy as np
import pytest

import oracle
import synth
from tests.test_gpu_decode import check_step

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32_LEVEL = 1e-4  # max |dlogit| / max |oracle logit| of the tensor-core path (exact int8 operands, split activations)


@pytest.fixture(scope="module")
def tqd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import token_quantized_decode_gb300 as t
    return t


def decode_vs_oracle(dec, om, tok, pos, n, seq=0):
    worst = 0.0
    for i in range(n):
        ref_tok, ref_lg = om.step(tok, pos)
        got = dec.decode_step(tok, pos, seq=seq)
        worst = max(worst, check_step(dec.logits(seq=seq), got, ref_lg, ref_tok, f"decode step {i} pos {pos}"))
        tok, pos = ref_tok, pos + 1
    return worst


@pytest.mark.parametrize("P", [1, 7, 16, 17, 40])
def test_prefill_tiles_tiny(tqd, P):
    """P = 1 (one slot), 7 (one partial tile), 16 (one full tile), 17 (a full
    tile, then a one-slot tile), 40 (two full tiles and a ragged one), on a
    one-sequence model; then three teacher-forced decode steps."""
    cfg = synth.TINY
    model = synth.make_model(cfg, 4)
    ids = synth.token_ids(1000, 7, P, cfg.vocab)
    om = oracle.OracleModel(model, P + 4)
    tok, lg = om.prefill(ids)
    dec = tqd.Decoder(model, P + 4, 1)
    got = dec.prefill_batch(ids)
    worst = check_step(dec.logits(), got, lg, tok, "prefill tiles")
    assert dec.next_pos() == P
    worst = max(worst, decode_vs_oracle(dec, om, tok, P, 3))
    assert worst < F32_LEVEL
    dec.close()


def test_prefill_tiles_continue_at_an_offset_then_batched_decode(tqd):
    """Sequence 2 of a four-sequence bf16 model (no QK-norm): 9 positions, then
    21 more from position 9 (tiles off the 16-position grid); sequences 0, 1
    and 3 stay empty.  Then one batched step of sequences 0-2 (two at position
    0, one at 30) against the oracle."""
    cfg = synth.ModelConfig(2, 256, 6, 2, 64, 768, 4096, False, "bf16", 1e5)
    model = synth.make_model(cfg, 6)
    a = synth.token_ids(1000, 3, 9, cfg.vocab)
    b = synth.token_ids(1000, 4, 21, cfg.vocab)
    om = oracle.OracleModel(model, 40)
    om.prefill(a)
    tok, lg = om.prefill(b, start=9)
    dec = tqd.Decoder(model, 40, 4)
    dec.prefill_batch(a, seq=2)
    got = dec.prefill_batch(b, seq=2)
    worst = check_step(dec.logits(seq=2), got, lg, tok, "second prefill")
    assert dec.next_pos(seq=2) == 30
    assert all(dec.next_pos(seq=s) == 0 for s in (0, 1, 3))
    firsts = [int(synth.token_ids(1000, 50 + s, 1, cfg.vocab)[0]) for s in (0, 1)]
    refs = []
    for s in (0, 1):
        o = oracle.OracleModel(model, 4)
        refs.append(o.step(firsts[s], 0))
    refs.append(om.step(tok, 30))
    nxt = dec.decode_step_batch(np.array(firsts + [tok]), np.array([0, 0, 30]))
    for s in range(3):
        worst = max(worst, check_step(dec.logits(seq=s), int(nxt[s]), refs[s][1], refs[s][0], f"batched seq {s}"))
    assert worst < F32_LEVEL
    dec.close()


def test_prefill_tiles_match_the_stepwise_prefill(tqd):
    """The same 37-position prompt prefilled position by position (persistent
    kernel) and in tiles: equal next tokens, logits equal to f32 level, and the
    same logits after three decode steps fed identical tokens (so the two
    caches hold the same rows)."""
    cfg = synth.TINY
    model = synth.make_model(cfg, 8)
    ids = synth.token_ids(1000, 9, 37, cfg.vocab)
    step = tqd.Decoder(model, 48, 1, tqd.TQD_SCHED_PERSISTENT)
    tile = tqd.Decoder(model, 48, 1, tqd.TQD_SCHED_PERSISTENT)
    ts, tt = step.prefill(ids), tile.prefill_batch(ids)
    ls, lt = step.logits(), tile.logits()
    assert ts == tt
    assert np.max(np.abs(lt - ls)) <= 1e-5 * np.max(np.abs(ls))
    tok, pos = ts, 37
    for _ in range(3):
        a = step.decode_step(tok, pos)
        tile.decode_step(tok, pos)
        ls, lt = step.logits(), tile.logits()
        assert np.max(np.abs(lt - ls)) <= 1e-5 * np.max(np.abs(ls))
        tok, pos = a, pos + 1
    step.close()
    tile.close()


def test_prefill_tiles_refusals(tqd):
    model = synth.make_model(synth.TINY, 0)
    dec = tqd.Decoder(model, 20, 1)
    with pytest.raises(tqd.TQDError) as ei:
        dec.prefill_batch(np.arange(21) % 7)
    assert ei.value.name == "TQD_ERR_CAPACITY"
    with pytest.raises(tqd.TQDError) as ei:
        dec.prefill_batch([1, 2, synth.TINY.vocab])
    assert ei.value.name == "TQD_ERR_BAD_ARG"
    with pytest.raises(tqd.TQDError) as ei:
        dec.prefill_batch([])
    assert ei.value.name == "TQD_ERR_BAD_ARG"
    assert dec.next_pos() == 0
    # the refusals left the sequence usable
    om = oracle.OracleModel(model, 20)
    assert dec.prefill_batch([3, 4, 5]) == om.prefill([3, 4, 5])[0]
    assert dec.next_pos() == 3
    dec.close()
    # eight query heads per kv head: the single-sequence path runs it, the
    # batched kernels (at most four) do not
    wide = synth.ModelConfig(1, 256, 8, 1, 64, 512, 4096, True, "q8_0", 1e6)
    dw = tqd.Decoder(synth.make_model(wide, 0), 8, 1)
    with pytest.raises(tqd.TQDError) as ei:
        dw.prefill_batch([1, 2])
    assert ei.value.name == "TQD_ERR_UNSUPPORTED_CONFIG"
    assert dw.prefill([1, 2]) >= 0
    dw.close()
