#!/usr/bin/env python
"""Batch-1 greedy decode throughput of the Qwen3-0.6B-shape Q8_0 workload
(511-token prompt prefilled, then greedy decode steps at positions 511..638)
on GB300, against the HBM roofline, with the oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tqd|reference]

A step is one decode token: embed, 28 layers, final norm, lm_head, argmax.
Timed tokens run as device-chained windows of up to 128 tokens starting at
position 511 (the sequence is truncated back to the prompt between windows,
outside the timed region).  Inputs are resident in HBM; every token streams
~766 MB of weights and KV, more than the 129 MB L2, so no L2 flush is needed.
Multi-GPU runs are independent replicas (one model per GPU, no collective).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "batch-1 decode tokens/sec (Qwen3-0.6B-shape Q8_0) and % of HBM roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "qwen3_0.6b"


def metric_for(wl) -> str:
    """The headline metric on the default workload; the other workloads
    (parity cases, measured on request) say which workload they are."""
    if wl.name == synth.WORKLOADS[DEFAULT_WORKLOAD].name:
        return METRIC
    return f"decode tokens/sec, all sequences ({wl.name}) and % of HBM roofline"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=4096, help="timed decode tokens")
    p.add_argument("--warmup", type=int, default=256, help="untimed decode tokens first")
    p.add_argument("--impl", choices=["tqd", "reference"], default="tqd")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    p.add_argument("--schedule", choices=["persistent", "graph"], default="persistent")
    p.add_argument("--e2e-steps", type=int, default=128)
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample length")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--kv-source", choices=["prefill", "upload"], default="prefill",
                   help="prefill the prompt on the GPU, or upload a seeded stand-in KV history of the same "
                        "length (for profiling captures that should not include the prefill launches)")
    p.add_argument("--prefill", choices=["tiles", "steps"], default="tiles",
                   help="prefill in tiles of 16 positions (tqd_prefill_batch) or position by position "
                        "(tqd_prefill); batch-1 runs time both after the decode measurement")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_traffic(bytes_per_launch: float):
    """DRAM bytes per launch: the committed ncu capture's ratio of DRAM traffic
    to algorithmic bytes times this launch's algorithmic bytes, or None when
    the kernel sources changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "k_persist_qwen3-0.6b_traffic.txt")
    try:
        kv = {}
        for line in open(path):
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
        h = hashlib.sha256()
        for f in kv["sources"].split():
            h.update(open(os.path.join(ROOT, "token_quantized_decode_gb300", "csrc", f), "rb").read())
        if h.hexdigest() != kv["sources_sha256"]:
            return None
        return float(kv["traffic_over_algorithmic"]) * bytes_per_launch
    except Exception:
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, _, r in rows:
            for n, v in zip(names, r[1:]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [r[0] for r in rows] if rows else []
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ oracle baseline

def oracle_sample(wl, seconds: float, max_steps: int | None = None):
    """Oracle decode steps at the workload's shape after a seeded stand-in KV
    history of prompt_len rows (no oracle prefill); returns (tok/s, steps,
    threads, seconds)."""
    import oracle
    cfg = wl.model
    model = synth.make_model(cfg, wl.model_seed)
    k, v = synth.kv_fill(cfg, 7, 0, wl.prompt_len, -1.0, 1.0)
    om = oracle.OracleModel(model, wl.prompt_len + wl.decode_steps)
    om.kv_load(k, v)
    del k, v
    tok, pos, n = int(synth.prompt(wl)[-1]), wl.prompt_len, 0
    t0 = time.perf_counter()
    while True:
        tok, _ = om.step(tok, pos)
        pos += 1
        n += 1
        el = time.perf_counter() - t0
        if (max_steps is not None and n >= max_steps) or (max_steps is None and el >= seconds) \
                or pos >= wl.prompt_len + wl.decode_steps:
            break
    return n / el, n, oracle.max_threads(), el


# ------------------------------------------------------------------ distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value: float) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, value: float) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ arms

def run_reference(args, wl, world, rank):
    if rank != 0:
        return None
    # warm-up steps, then K timed oracle steps on the host cores
    if args.warmup:
        oracle_sample(wl, 0, max_steps=min(args.warmup, 3))
    k = max(1, min(args.steps, wl.decode_steps))
    tps, n, cores, el = oracle_sample(wl, 0, max_steps=k)
    sample = (f"{n} oracle decode steps at positions {wl.prompt_len}..{wl.prompt_len + n - 1} after a "
              f"seeded stand-in KV history of {wl.prompt_len} rows (no oracle prefill)")
    line = {
        "impl": "reference", "metric": metric_for(wl), "value": tps, "unit": UNIT, "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": 1000.0 * el / n, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "prompt_len": wl.prompt_len, "batch": wl.batch},
        "cpu_baseline": {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": tps, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def prefill(dec, ids, seq, tiles):
    """The prompt through tqd_prefill_batch (tiles), or tqd_prefill where the
    shape has no batched step or steps were asked for."""
    import token_quantized_decode_gb300 as tqd
    if tiles:
        try:
            return dec.prefill_batch(ids, seq=seq)
        except tqd.TQDError as e:
            if e.name != "TQD_ERR_UNSUPPORTED_CONFIG":
                raise
    return dec.prefill(ids, seq=seq)


def time_prefill(dec, wl, stream, kv_pos, w_and_row, emb_row):
    """Prompt throughput of one sequence's prefill through the C ABI (prompt
    upload and next-token readback included): tiles (median of 3 after one
    warm-up call that instantiates the tile graphs) and position by position
    (one call).  Algorithmic bytes of the tiled prefill: per tile, the layers'
    weights once, one embedding row per position, the K/V rows the tile
    attends to (each once) and the rows it writes; the lm_head once."""
    import torch
    import token_quantized_decode_gb300 as tqd
    cfg, P = wl.model, wl.prompt_len
    ids = synth.prompt(wl, seq=0)

    def once(fn):
        dec.truncate(0)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn(ids)
        e.record(stream)
        torch.cuda.synchronize()
        return s.elapsed_time(e)

    try:
        once(dec.prefill_batch)
    except tqd.TQDError as e:
        if e.name != "TQD_ERR_UNSUPPORTED_CONFIG":
            raise
        return None
    tiles_ms = float(np.median([once(dec.prefill_batch) for _ in range(3)]))
    steps_ms = once(dec.prefill)
    row_h = cfg.hidden * 17 // 16 if cfg.weight_type == "q8_0" else 2 * cfg.hidden
    head = cfg.vocab * row_h + 4 * cfg.hidden                  # lm_head rows + final norm
    layers = w_and_row - emb_row - head
    nbytes, p0 = head, 0
    while p0 < P:
        n = min(16, P - p0)
        nbytes += layers + n * emb_row + kv_pos * (p0 + n) + kv_pos * n
        p0 += n
    hbm, kind = peaks()
    return {"value": P / (tiles_ms / 1000.0), "unit": "prompt tokens/s", "tokens": P,
            "ms": tiles_ms, "tiles": (P + 15) // 16, "api": "tqd_prefill_batch (tiles of 16 positions)",
            "roofline_frac": nbytes / (tiles_ms / 1000.0) / 1e9 / hbm, "algorithmic_bytes": nbytes,
            "peak_kind": f"{kind} copy bandwidth",
            "stepwise": {"value": P / (steps_ms / 1000.0), "ms": steps_ms, "api": "tqd_prefill (one decode step per position)"}}


SAMPLING = dict(temperature=0.8, top_k=40, top_p=0.95, min_p=0.02, repeat_penalty=1.1, seed=1234)


def time_sampling(dec, wl, stream, firsts, greedy_ms):
    """Decode steps with a seeded draw after each (tqd_generate_sampled, or
    the batched form), timed like the greedy window: tokens/s and the added
    time per step against the greedy steps."""
    import torch
    import token_quantized_decode_gb300 as tqd
    P, D, B = wl.prompt_len, wl.decode_steps, wl.batch
    params = tqd.sampling(**SAMPLING)

    def window():
        for b in range(B):
            dec.truncate(P, seq=b)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        if B == 1:
            dec.generate_sampled(firsts[0], D, params)
        else:
            dec.generate_batch_sampled(np.array(firsts), D, params)
        e.record(stream)
        torch.cuda.synchronize()
        return s.elapsed_time(e)

    window()
    ms = float(np.median([window() for _ in range(3)]))
    return {"value": D * B / (ms / 1000.0), "unit": UNIT, "controls": SAMPLING, "ms_per_step": ms / D,
            "added_ms_per_step": ms / D - greedy_ms,
            "api": "tqd_generate_sampled" if B == 1 else "tqd_generate_batch_sampled",
            "note": ("after each step, one block per 1024-entry vocabulary slice and sequence keeps the "
                     "slice's top_k, then one block per sequence merges them and draws; steps launched one by one")}


def time_kv16(args, wl, model, stream, hbm, kind):
    """The same decode windows on a model whose KV cache holds f16 elements
    (TQD_KV_F16: rows rounded to binary16 as they are appended), after the
    same prompts prefilled in tiles (or the same history uploaded):
    tokens/s and the step's algorithmic bytes with two-byte K/V elements.
    Batch 1 runs the persistent schedule."""
    import torch
    import token_quantized_decode_gb300 as tqd
    cfg, P, D, B = wl.model, wl.prompt_len, wl.decode_steps, wl.batch
    schedule = tqd.TQD_SCHED_PERSISTENT if B == 1 else tqd.TQD_SCHED_GRAPH
    dec = tqd.Decoder(model, P + D, B, schedule, stream=stream, kv_type=tqd.TQD_KV_F16)
    if args.kv_source == "upload":
        firsts = []
        for b in range(B):
            k, v = synth.kv_fill(cfg, 7, b, P, -1.0, 1.0)
            dec.kv_upload(k, v, seq=b)
            del k, v
            firsts.append(int(synth.prompt(wl, seq=b)[-1]))
    else:
        firsts = [dec.prefill_batch(synth.prompt(wl, seq=b), seq=b) for b in range(B)]
    kv_pos = 2 * cfg.kv_width * 2 * cfg.n_layers
    w_and_row = dec.step_bytes(0) - 2 * kv_pos
    emb_row = cfg.hidden * 17 // 16 if cfg.weight_type == "q8_0" else 2 * cfg.hidden

    def window():
        for b in range(B):
            dec.truncate(P, seq=b)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        if B == 1:
            dec.generate(firsts[0], D)
        else:
            dec.generate_batch(np.array(firsts), D)
        e.record(stream)
        torch.cuda.synchronize()
        return s.elapsed_time(e)

    window()
    ms = float(np.median([window() for _ in range(5)]))
    nbytes = sum(w_and_row + (B - 1) * emb_row + B * kv_pos * (p + 2) for p in range(P, P + D)) / D
    dec.close()
    return {"value": D * B / (ms / 1000.0), "unit": UNIT, "ms_per_step": ms / D,
            "step_roofline_frac": nbytes / (hbm * 1e9) / (ms / D / 1000.0), "bytes_per_step": nbytes,
            "peak_kind": f"{kind} copy bandwidth",
            "api": ("tqd_generate" if B == 1 else "tqd_generate_batch") + " on a TQD_KV_F16 model (history "
                   + ("uploaded" if args.kv_source == "upload" else "prefilled in tiles") + ")"}


def run_tqd(args, wl, world, rank, local, pg):
    import torch
    import token_quantized_decode_gb300 as tqd

    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    cfg = wl.model
    model = synth.make_model(cfg, wl.model_seed)
    P, D, B = wl.prompt_len, wl.decode_steps, wl.batch
    schedule = tqd.TQD_SCHED_PERSISTENT if args.schedule == "persistent" else tqd.TQD_SCHED_GRAPH
    dec = tqd.Decoder(model, P + D, B, schedule, stream=stream)
    if B == 1 and P < 4096:
        del model
    firsts = []
    for b in range(B):
        ids = synth.prompt(wl, seq=b)
        if args.kv_source == "prefill":
            firsts.append(prefill(dec, ids, b, args.prefill == "tiles"))
        else:
            k, v = synth.kv_fill(cfg, 7, b, P, -1.0, 1.0)
            dec.kv_upload(k, v, seq=b)
            del k, v
            firsts.append(int(ids[-1]))
    first = firsts[0]
    kv_pos = 4 * cfg.kv_width * 2 * cfg.n_layers          # K and V bytes of one position, all layers
    w_and_row = dec.step_bytes(0) - 2 * kv_pos              # weights + one embedding row
    emb_row = cfg.hidden * 17 // 16 if cfg.weight_type == "q8_0" else 2 * cfg.hidden

    def step_bytes(p):
        """Algorithmic bytes of one step at position p for all B sequences:
        weights once, one embedding row and (p + 2) K/V positions per sequence."""
        return w_and_row + (B - 1) * emb_row + B * kv_pos * (p + 2)

    def windows(n_steps, at_least=1):
        """Window lengths summing to n_steps: at least `at_least` windows (when
        there are that many steps), none longer than the D decode positions."""
        k = max(at_least, -(-n_steps // D))
        k = min(k, n_steps)
        return [n_steps // k + (1 if i < n_steps % k else 0) for i in range(k)]

    def run_window(n):
        for b in range(B):
            dec.truncate(P, seq=b)
        if B == 1:
            dec.generate(first, n)
        else:
            dec.generate_batch(np.array(firsts), n)

    steps_timed = max(1, args.steps // B)   # --steps counts tokens (all sequences)
    for n in windows(max(1, args.warmup // B)):
        run_window(n)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ev = []
    barrier(pg)
    torch.cuda.synchronize()
    total_bytes = 0
    launches = 0
    for n in windows(steps_timed, at_least=5):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for b in range(B):
            dec.truncate(P, seq=b)
        s.record(stream)
        if B == 1:
            dec.generate(first, n)
        else:
            dec.generate_batch(np.array(firsts), n)
        e.record(stream)
        ev.append((s, e, n))
        total_bytes += sum(step_bytes(p) for p in range(P, P + n))
        if B > 1:
            launches += n * -(-B // 16) * (1 + 5 * cfg.n_layers + 1)  # one graph per group of 16 sequences
        else:
            launches += 1 if schedule == tqd.TQD_SCHED_PERSISTENT else n * dec.phase_count
    torch.cuda.synchronize()
    barrier(pg)
    clocks = sampler.stop()
    t_ms = sum(s.elapsed_time(e) for s, e, _ in ev)
    steps = sum(n for _, _, n in ev)
    win_rates = [n * B / (s.elapsed_time(e) / 1000.0) for s, e, n in ev]
    longest = max(n for _, _, n in ev)
    tokens = steps * B
    t_max = max_over_ranks(pg, t_ms)
    all_tokens = sum_over_ranks(pg, tokens)
    value = all_tokens / (t_max / 1000.0)
    per_launch_bytes = total_bytes / len(ev)
    per_launch_ms = t_ms / len(ev)

    # end to end through the C ABI: one decode call per step, host tokens in,
    # host tokens out, the host round trip inside the timed region
    for b in range(B):
        dec.truncate(P, seq=b)
    torch.cuda.synchronize()
    toks, pos = list(firsts), P
    n_e2e = min(args.e2e_steps, D)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        if B == 1:
            toks = [dec.decode_step(toks[0], pos)]
        else:
            toks = list(dec.decode_step_batch(np.array(toks), np.full(B, pos)))
        pos += 1
    e2e_s = time.perf_counter() - t0
    e2e_val = sum_over_ranks(pg, n_e2e * B) / max_over_ranks(pg, e2e_s)

    sampling_line = time_sampling(dec, wl, stream, firsts, t_max / steps)
    prefill_line = (time_prefill(dec, wl, stream, kv_pos, w_and_row, emb_row)
                    if B == 1 and args.kv_source == "prefill" else None)

    hbm, kind = peaks()
    achieved = per_launch_bytes / (per_launch_ms / 1000.0) / 1e9
    mean_step_bytes = total_bytes / steps
    persistent_b1 = B == 1 and schedule == tqd.TQD_SCHED_PERSISTENT
    if persistent_b1:
        kernel = "k_persist<%s>" % ("Q8_0" if cfg.weight_type == "q8_0" else "bf16")
    elif B > 1:
        kernel = "whole batched step (graph: tcgen05 matmuls + streaming attention)"
    else:
        kernel = "whole step (graph schedule)"
    line = {
        "metric": metric_for(wl), "value": value, "unit": UNIT, "n_gpus": world, "steps": tokens,
        "warmup": args.warmup, "ms_per_step": t_max / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "prompt_len": P, "decode_positions": f"{P}..{P + longest - 1}",
                   "timed_windows": len(ev),
                   "batch": B, "schedule": args.schedule if B == 1 else "batched graph",
                   "weights": ("Q8_0 (34-byte blocks)" if cfg.weight_type == "q8_0" else "bf16") + ", resident",
                   "kv_history": args.kv_source + (f" ({args.prefill})" if args.kv_source == "prefill" else ""),
                   "l2": "inputs larger than L2: each step streams %.0f MB vs 129 MB L2" % (mean_step_bytes / 1e6),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm,
                     "traffic": (measured_traffic(per_launch_bytes)
                                 if persistent_b1 and wl.name.startswith("qwen3-0.6b-shape-q8_0-prompt511")
                                 else None),
                     "kernel": kernel, "bytes_per_launch": per_launch_bytes, "ms_per_launch": per_launch_ms,
                     "peak_kind": f"{kind} copy bandwidth"},
        "step_roofline_frac": (mean_step_bytes / (hbm * 1e9)) / (t_max / steps / 1000.0),
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": 4 * B,
                "d2h_bytes_per_step": 16 if persistent_b1 else (4 + 16) * B,
                "api": "tqd_decode_step per token" if B == 1 else "tqd_decode_step_batch per step",
                "copies": ("the token as a launch argument; the next token inside the 16-byte state record read back"
                           if persistent_b1 else "the tokens up, the next tokens and the state records back")},
        "windows": {"n": len(ev), "steps_each": sorted({n for _, _, n in ev}),
                    "median": float(np.median(win_rates)), "min": float(min(win_rates)),
                    "max": float(max(win_rates)), "unit": UNIT,
                    "note": "each window restarts at the prompt's end; value is all timed tokens over the summed window times"},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    line["sampling"] = sampling_line
    if prefill_line:
        line["prefill"] = prefill_line
    dec.close()
    if B > 1 or P >= 4096:  # the workloads where the K/V bytes rival the weights
        line["kv_f16"] = time_kv16(args, wl, model, stream, hbm, kind)
    return line


def main():
    args = parse()
    wl = synth.WORKLOADS[args.workload]
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        line = run_reference(args, wl, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    line = run_tqd(args, wl, world, rank, local, pg)
    if rank == 0:
        if not args.no_cpu_baseline:
            import oracle
            tps, n, cores, el = oracle_sample(wl, args.cpu_seconds)
            line["cpu_baseline"] = {
                "value": tps, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": (f"{n} oracle decode steps ({el:.1f} s) at positions {wl.prompt_len}.. after a seeded "
                           f"stand-in KV history of {wl.prompt_len} rows")}
            oracle.set_threads(1)
            tps1, n1, _, el1 = oracle_sample(wl, min(args.cpu_seconds, 4.0))
            oracle.set_threads(cores)
            line["cpu_baseline"]["one_core"] = {
                "value": tps1, "unit": UNIT, "cores": 1,
                "sample": f"{n1} oracle decode steps ({el1:.1f} s) on one thread, same positions"}
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
