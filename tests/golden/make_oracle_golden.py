"""Writes oracle_tiny.txt: the oracle's greedy run on the tiny Qwen3-shaped
workload (2 layers, hidden 256, seed 0, 32-token prompt from seed 1000, 16
generated tokens).  Calls only the oracle and the input generator; the stored
values pin the oracle against regressions and across host architectures."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402


def run():
    wl = synth.WORKLOADS["tiny"]
    m = synth.make_model(wl.model, wl.model_seed)
    ids = synth.prompt(wl)
    om = oracle.OracleModel(m, wl.prompt_len + wl.decode_steps + 1)
    nxt, logits = om.prefill(ids)
    toks, sums, maxes = [nxt], [float(logits.sum())], [float(np.abs(logits).max())]
    pos = wl.prompt_len
    for _ in range(wl.decode_steps - 1):
        nxt, logits = om.step(nxt, pos)
        pos += 1
        toks.append(nxt)
        sums.append(float(logits.sum()))
        maxes.append(float(np.abs(logits).max()))
    return ids, toks, sums, maxes


if __name__ == "__main__":
    ids, toks, sums, maxes = run()
    with open(os.path.join(HERE, "oracle_tiny.txt"), "w") as f:
        f.write("# written by make_oracle_golden.py (oracle only)\n")
        f.write("prompt " + " ".join(map(str, ids)) + "\n")
        f.write("tokens " + " ".join(map(str, toks)) + "\n")
        f.write("logit_sums " + " ".join(repr(s) for s in sums) + "\n")
        f.write("logit_absmax " + " ".join(repr(s) for s in maxes) + "\n")
