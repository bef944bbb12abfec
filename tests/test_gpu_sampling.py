"""The device sampler (tqd_sample, tqd_generate_sampled,
tqd_generate_batch_sampled) against the sampling oracle, on the logits the
device itself produced (the oracle takes them as input).  Kept sets that
f32 values decide (penalties, temperature, top_k, min_p) agree exactly; the
masses of top_p and the draw are the device's fixed-point sums, so a token
must equal the oracle's wherever the oracle's decisive masses lie farther
than MARGIN from their thresholds, and be in the oracle's kept set
otherwise."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from oracle import sampling as S

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MARGIN = 1e-5  # relative mass distance beyond which a draw is unique

PARAMS = [
    dict(temperature=1.0),
    dict(temperature=0.7, top_k=40),
    dict(temperature=1.3, top_p=0.9),
    dict(temperature=1.0, top_k=50, top_p=0.8, min_p=0.05),
    dict(temperature=0.9, min_p=0.1),
    dict(temperature=1.0, top_k=1),
    dict(temperature=1.1, repeat_penalty=1.3, presence_penalty=0.4, frequency_penalty=0.2),
    dict(temperature=0.8, top_k=200, top_p=0.95, repeat_penalty=0.7, frequency_penalty=-0.3),
    dict(temperature=2.0, top_p=0.5),
    dict(temperature=0.05, top_p=0.99),
]


@pytest.fixture(scope="module")
def tqd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import token_quantized_decode_gb300 as t
    return t


def oracle_kw(p):
    return dict(temperature=p.get("temperature", 1.0), top_k=p.get("top_k", 0), top_p=p.get("top_p", 1.0),
                min_p=p.get("min_p", 0.0), repeat=p.get("repeat_penalty", 1.0),
                presence=p.get("presence_penalty", 0.0), frequency=p.get("frequency_penalty", 0.0))


def check_draw(got, logits, history, pos, p, seed, where):
    """got must be the oracle's token, or a kept token where a rounding could decide."""
    kw = oracle_kw(p)
    want, margin = S.sample(logits, history, pos, seed=seed, **kw)
    if margin > MARGIN:
        assert got == want, f"{where}: token {got} != oracle {want} (margin {margin:.2e})"
        return 1
    if kw["temperature"] > 0:
        _, keep, _ = S.kept(logits, history, **kw)
        assert keep[got], f"{where}: token {got} outside the kept set"
    return 0


def history_prompt(V):
    """A prompt with repeated tokens, so counts above one reach the penalties."""
    base = synth.token_ids(1000, 21, 12, V)
    return np.concatenate([base, base[:5], base[:2], [base[0]] * 3]).astype(np.int32)


def test_sample_matches_the_oracle(tqd):
    cfg = synth.TINY
    model = synth.make_model(cfg, 12)
    ids = history_prompt(cfg.vocab)
    P = len(ids)
    dec = tqd.Decoder(model, P + 2, 1)
    dec.prefill(ids)
    logits = dec.logits()
    unique = 0
    for i, p in enumerate(PARAMS):
        for seed in range(12):
            got = dec.sample(tqd.sampling(seed=1000 * i + seed, **p))
            unique += check_draw(got, logits, ids, P, p, 1000 * i + seed, f"params {i} seed {seed}")
    # the tiny model's logits are flat (one token ~ 1/4096 of the mass) and one
    # top_p boundary here lies within 4e-7 of its threshold: most draws, not all,
    # are unique
    assert unique >= 0.8 * len(PARAMS) * 12
    assert np.array_equal(dec.logits(), logits)  # drawing reads the logits, never writes them
    # after draws replaced it, temperature 0 gives the greedy token of the logits again
    assert dec.sample(tqd.sampling(temperature=0.0)) == S.greedy(logits)
    dec.close()


def test_greedy_rules(tqd):
    """temperature <= 0 and top_k = 1 (neutral penalties) give the greedy
    sequence exactly, on both schedules."""
    cfg = synth.TINY
    model = synth.make_model(cfg, 13)
    ids = synth.token_ids(1000, 3, 9, cfg.vocab)
    for schedule in (tqd.TQD_SCHED_GRAPH, tqd.TQD_SCHED_PERSISTENT):
        dec = tqd.Decoder(model, 40, 1, schedule)
        first = dec.prefill(ids)
        greedy = dec.generate(first, 12)
        for p in (dict(temperature=0.0, top_k=7, seed=3), dict(temperature=-1.0),
                  dict(temperature=0.8, top_k=1, seed=5), dict(temperature=1.7, top_k=1, top_p=0.3, seed=6)):
            dec.truncate(len(ids))
            got = dec.generate_sampled(first, 12, tqd.sampling(**p))
            assert np.array_equal(got, greedy), p
        dec.close()


@pytest.mark.parametrize("schedule", ["graph", "persistent"])
def test_generate_sampled_is_the_chained_draw(tqd, schedule):
    """Twelve device-chained sampled steps; replayed step by step on a second
    decoder fed the chain's tokens, each drawn token is the oracle's draw from
    that step's logits at its position with the inputs so far as history."""
    cfg = synth.TINY
    model = synth.make_model(cfg, 14)
    ids = history_prompt(cfg.vocab)
    P, n = len(ids), 12
    sched = tqd.TQD_SCHED_GRAPH if schedule == "graph" else tqd.TQD_SCHED_PERSISTENT
    p = dict(temperature=0.9, top_k=60, top_p=0.92, repeat_penalty=1.2, frequency_penalty=0.1)
    chain = tqd.Decoder(model, P + n + 1, 1, sched)
    first = chain.prefill(ids)
    got = chain.generate_sampled(first, n, tqd.sampling(seed=77, **p))
    assert chain.next_pos() == P + n
    replay = tqd.Decoder(model, P + n + 1, 1, sched)
    replay.prefill(ids)
    hist = list(ids)
    tok = first
    for i in range(n):
        replay.decode_step(tok, P + i)
        hist.append(tok)
        check_draw(int(got[i]), replay.logits(), hist, P + i + 1, p, 77, f"step {i}")
        tok = int(got[i])
    chain.close()
    replay.close()


def test_generate_batch_sampled(tqd):
    """Four sequences, six batched sampled steps, replayed with single batched
    steps fed the chain's tokens."""
    cfg = synth.TINY
    model = synth.make_model(cfg, 15)
    n_seq, n, P = 4, 6, 10
    p = dict(temperature=1.2, top_p=0.85, presence_penalty=0.3)
    prompts = [synth.token_ids(1000, 30 + b, P, cfg.vocab) for b in range(n_seq)]
    chain = tqd.Decoder(model, P + n + 1, n_seq)
    replay = tqd.Decoder(model, P + n + 1, n_seq)
    firsts = [chain.prefill(prompts[b], seq=b) for b in range(n_seq)]
    for b in range(n_seq):
        replay.prefill(prompts[b], seq=b)
    got = chain.generate_batch_sampled(np.array(firsts), n, tqd.sampling(seed=5, **p))
    hists = [list(prompts[b]) for b in range(n_seq)]
    toks = list(firsts)
    for i in range(n):
        replay.decode_step_batch(np.array(toks), np.full(n_seq, P + i))
        for b in range(n_seq):
            hists[b].append(toks[b])
            check_draw(int(got[i, b]), replay.logits(seq=b), hists[b], P + i + 1, p, 5, f"step {i} seq {b}")
        toks = [int(t) for t in got[i]]
    chain.close()
    replay.close()


def test_planted_ties_and_an_odd_vocabulary(tqd):
    """3000 lm_head rows copied from the argmax row: at least 3000 exactly equal
    largest logits, so top_k and top_p boundaries fall inside a tie (a value bin too
    full to sort, then ties in index order).  Vocabulary 4093 (not a multiple
    of the scan's four elements per thread)."""
    cfg = dataclasses.replace(synth.TINY, vocab=4093)
    model = synth.make_model(cfg, 16)
    ids = np.array([5, 17, 42, 3500, 4000, 60, 99], dtype=np.int32)  # no token in [100, 3100)
    dec = tqd.Decoder(model, 16, 1)
    dec.prefill(ids)
    r = int(np.argmax(dec.logits()))
    dec.close()
    lm = model.lm_head.copy()
    lm[100:3100] = lm[r]
    model = dataclasses.replace(model, lm_head=lm)
    dec = tqd.Decoder(model, 16, 1)
    dec.prefill(ids)
    logits = dec.logits()
    top = logits.max()
    assert np.count_nonzero(logits == top) >= 3000
    cases = [dict(temperature=1.0, top_k=1), dict(temperature=1.0, top_k=50), dict(temperature=1.0, top_k=2500),
             dict(temperature=0.5, top_p=0.3), dict(temperature=1.0, top_k=3050, top_p=0.6),
             dict(temperature=1.0, min_p=0.5)]
    for i, p in enumerate(cases):
        for seed in range(6):
            got = dec.sample(tqd.sampling(seed=seed, **p))
            check_draw(got, logits, ids, len(ids), p, seed, f"case {i} seed {seed}")
    dec.close()


def test_qwen3_vocabulary(tqd):
    """The full 151,936-token vocabulary of the Qwen3 shape, after an
    eight-token prompt prefilled in one tile."""
    wl = synth.WORKLOADS["qwen3_0.6b"]
    model = synth.make_model(wl.model, wl.model_seed)
    ids = synth.prompt(wl)[:8]
    dec = tqd.Decoder(model, 16, 1, tqd.TQD_SCHED_PERSISTENT)
    dec.prefill_batch(ids)
    logits = dec.logits()
    for i, p in enumerate(PARAMS):
        for seed in range(3):
            got = dec.sample(tqd.sampling(seed=seed, **p))
            check_draw(got, logits, ids, len(ids), p, seed, f"params {i} seed {seed}")
    dec.close()


def test_sampling_refusals(tqd):
    model = synth.make_model(synth.TINY, 0)
    dec = tqd.Decoder(model, 16, 1)
    with pytest.raises(tqd.TQDError) as ei:
        dec.sample(tqd.sampling())
    assert ei.value.name == "TQD_ERR_NOT_PREFILLED"
    dec.prefill([1, 2, 3])
    for bad in (dict(top_p=0.0), dict(top_p=1.5), dict(min_p=2.0), dict(min_p=-0.1), dict(repeat_penalty=0.0),
                dict(top_k=-1), dict(temperature=float("nan")), dict(presence_penalty=float("inf"))):
        with pytest.raises(tqd.TQDError) as ei:
            dec.sample(tqd.sampling(**bad))
        assert ei.value.name == "TQD_ERR_BAD_ARG", bad
    assert 0 <= dec.sample(tqd.sampling(seed=1)) < synth.TINY.vocab
    dec.truncate(2)
    with pytest.raises(tqd.TQDError) as ei:
        dec.sample(tqd.sampling())
    assert ei.value.name == "TQD_ERR_NOT_PREFILLED"
    k, v = synth.kv_fill(synth.TINY, 1, 0, 4)
    dec.kv_upload(k, v)
    with pytest.raises(tqd.TQDError) as ei:
        dec.sample(tqd.sampling())
    assert ei.value.name == "TQD_ERR_NOT_PREFILLED"
    dec.close()


def op_draw(tqd, logits, hist, p, seed):
    """tqd_op_sample on caller tensors: the token drawn after `hist`."""
    from token_quantized_decode_gb300 import ops
    V = len(logits)
    lg = torch.tensor(np.asarray(logits, dtype=np.float32), device="cuda")
    toks = torch.tensor(list(hist) + [0], dtype=torch.int32, device="cuda")
    scratch = torch.empty(ops.tqd_sample_scratch_bytes(V), dtype=torch.uint8, device="cuda")
    ops.tqd_op_sample(lg, V, toks, len(hist), tqd.sampling(seed=seed, **p), scratch)
    torch.cuda.synchronize()
    return int(toks[-1].item())


def test_op_sample_matches_the_oracle(tqd):
    """The operator entry point on planted logits (a peaked distribution, so
    the draws are mostly unique) against the sampling oracle."""
    rng = np.random.default_rng(21)
    V = 1001
    unique = 0
    for i, p in enumerate(PARAMS):
        for seed in range(4):
            l = (rng.normal(size=V) * 3).astype(np.float32)
            hist = rng.integers(0, V, size=9)
            unique += check_draw(op_draw(tqd, l, hist, p, 100 * i + seed), l, hist, len(hist), p,
                                 100 * i + seed, f"params {i} seed {seed}")
    assert unique >= 0.8 * len(PARAMS) * 4


def test_top_k_one_is_greedy_where_the_temperature_merges_two_logits(tqd):
    """Two adjacent f32 logits l_lo < l_hi with l_lo / T == l_hi / T in f32,
    the lower index holding l_lo: top_k = 1 and a tiny top_p still give the
    greedy token, top_k = 2 keeps both."""
    T = 3.0
    t = np.float32(T)
    lo = np.float32(7.0)
    while np.float32(lo / t) != np.float32(np.nextafter(lo, np.float32(np.inf)) / t):
        lo = np.nextafter(lo, np.float32(np.inf))
    hi = np.nextafter(lo, np.float32(np.inf))
    rng = np.random.default_rng(22)
    for i in range(8):
        l = rng.normal(size=3000).astype(np.float32)
        a, b = sorted(rng.choice(3000, 2, replace=False))
        l[a], l[b] = lo, hi
        for seed in range(3):
            assert op_draw(tqd, l, [int(a)], dict(temperature=T, top_k=1), seed) == b
            assert op_draw(tqd, l, [1, 2], dict(temperature=T, top_p=1e-6), seed) == b
            assert op_draw(tqd, l, [3], dict(temperature=T, top_k=2), seed) in (a, b)


def test_an_overflowing_temperature_is_the_greedy_limit(tqd):
    """l_max / T beyond f32 (T = 1e-38, and negative logits at 1e-39): the
    greedy token of the penalised logits."""
    rng = np.random.default_rng(23)
    for i in range(6):
        l = (rng.normal(size=2000) * 4).astype(np.float32)
        hist = rng.integers(0, 2000, size=7)
        p = dict(temperature=1e-38, top_p=0.9, repeat_penalty=1.3, presence_penalty=0.2)
        want = S.greedy(S.penalised(l, hist, 1.3, 0.2, 0.0))
        assert S.sample(l, hist, len(hist), 1e-38, top_p=0.9, repeat=1.3, presence=0.2)[0] == want
        assert op_draw(tqd, l, hist, p, i) == want
    l = np.array([-3.0, -1.0, -2.0, -1.0, -5.0], dtype=np.float32)
    assert op_draw(tqd, l, [0], dict(temperature=1e-39), 1) == 1


def test_two_pass_draw_edges(tqd):
    """Draws with 1 <= top_k <= 64 take two passes (each 1024-token slice keeps
    its own first top_k, one block merges them).  Planted lm_head rows put the
    whole first top_k in one slice (the merge's threshold is then far below the
    boundary) or make every logit equal (the order is the index order across
    all slices; the penalised history tokens then move down the order);
    top_k = 64 is the last two-pass value and 65 the first one-pass value.
    The history avoids the planted rows (the lm_head is also the embedding), so
    planting leaves the hidden state alone.  Vocabulary 20011: twenty slices,
    the last one partial."""
    cfg = dataclasses.replace(synth.TINY, vocab=20011)
    base_model = synth.make_model(cfg, 21)
    ids = np.array([11, 250, 19000, 11, 5, 250, 11], dtype=np.int32)
    dec = tqd.Decoder(base_model, 16, 1)
    dec.prefill(ids)
    r = int(np.argmax(dec.logits()))
    dec.close()
    cases = [dict(temperature=1.0, top_k=40), dict(temperature=0.7, top_k=64, top_p=0.5),
             dict(temperature=1.0, top_k=65), dict(temperature=1.2, top_k=40, repeat_penalty=1.3),
             dict(temperature=0.9, top_k=20, min_p=0.3, presence_penalty=0.5), dict(temperature=1.0, top_k=1)]
    for planted in (slice(7000, 7070), slice(0, cfg.vocab)):
        lm = base_model.lm_head.copy()
        lm[planted] = lm[r]
        model = dataclasses.replace(base_model, lm_head=lm)
        dec = tqd.Decoder(model, 16, 1)
        dec.prefill(ids)
        logits = dec.logits()
        assert np.count_nonzero(logits == logits.max()) >= 70
        for i, p in enumerate(cases):
            for seed in range(5):
                got = dec.sample(tqd.sampling(seed=seed, **p))
                check_draw(got, logits, ids, len(ids), p, seed, f"rows {planted} case {i} seed {seed}")
        dec.close()
