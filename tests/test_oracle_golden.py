"""The oracle's greedy run on the tiny workload against the stored values
written by tests/golden/make_oracle_golden.py, and the cited page values."""
import os

import numpy as np

import oracle
import synth
from tests.golden.make_oracle_golden import run

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_kv(path):
    out = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if "=" in line:
            k, v = line.split("=", 1)
            out[k.strip()] = v.strip()
    return out


def test_tiny_greedy_run_matches_stored():
    rows = {}
    for line in open(os.path.join(HERE, "oracle_tiny.txt")):
        if line.startswith("#"):
            continue
        k, *vals = line.split()
        rows[k] = vals
    ids, toks, sums, maxes = run()
    assert list(map(int, rows["prompt"])) == list(map(int, ids))
    assert list(map(int, rows["tokens"])) == toks
    # libm (exp, pow, sin, cos) may differ in the last bit between hosts
    assert np.allclose(np.array(rows["logit_sums"], dtype=float), sums, rtol=1e-9, atol=1e-9)
    assert np.allclose(np.array(rows["logit_absmax"], dtype=float), maxes, rtol=1e-9)


def test_cited_page_values():
    g = load_kv(os.path.join(HERE, "p1_correctness_ladder.txt"))
    lo, hi = (int(b, 16) for b in g["q8_fabricated_scale_bytes"].split())
    assert oracle.f16_to_f64(lo | (hi << 8)) == float(g["q8_fabricated_scale_value"])
    assert g["argmax_case"].endswith("-> 140011")
    assert float(g["tol_q8_matvec"]) == 5e-4
    assert synth.QWEN3_06B.vocab == 151936
