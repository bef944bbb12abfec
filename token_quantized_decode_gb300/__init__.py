"""Python binding of libtqd, the GB300 (sm_103a) greedy decoder for
Qwen3-shaped models with Q8_0 or bf16 weights.

Every function here marshals arguments into one call of the C ABI of the
same name (include/tqd.h); all computation runs in the library's CUDA
kernels.  PyTorch is used only to hand device memory (tensor data pointers)
and streams to the operator entry points.
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._lib import (TQD_KV_F16, TQD_KV_F32, TQD_SCHED_GRAPH, TQD_SCHED_PERSISTENT, TQD_WEIGHT_BF16,
                   TQD_WEIGHT_Q8_0, TQDError,
                   check, lib, tqd_config, tqd_host_weights, tqd_layer_weights, tqd_sampling)

__all__ = [
    "TQDError", "TQD_SCHED_GRAPH", "TQD_SCHED_PERSISTENT", "TQD_WEIGHT_Q8_0", "TQD_WEIGHT_BF16", "TQD_KV_F32",
    "TQD_KV_F16",
    "make_config", "make_host_weights", "tqd_status_name", "tqd_create", "tqd_destroy", "tqd_reset",
    "tqd_truncate", "tqd_next_pos", "tqd_prefill", "tqd_prefill_batch", "tqd_kv_upload", "tqd_decode_step", "tqd_generate",
    "tqd_decode_step_batch", "tqd_generate_batch", "tqd_sample", "tqd_generate_sampled",
    "tqd_generate_batch_sampled", "sampling", "tqd_read_logits", "tqd_phase_count", "tqd_step_bytes",
    "Decoder",
]

_LAYER_FIELDS = ("attn_norm", "wq", "wk", "wv", "wo", "q_norm", "k_norm", "ffn_norm", "w_gate", "w_up",
                 "w_down")


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays passed to libtqd must be C-contiguous")
        return a.ctypes.data
    return int(a.data_ptr())  # torch tensor


def _stream(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def make_config(model_cfg, max_seq: int, max_batch: int = 1, schedule: int = TQD_SCHED_GRAPH,
                kv_type: int = TQD_KV_F32) -> tqd_config:
    """tqd_config from an object with the model's hyper-parameter fields
    (n_layers, hidden, n_heads, n_kv_heads, head_dim, intermediate, vocab,
    qk_norm, weight_type 'q8_0' | 'bf16', rope_theta, rms_eps)."""
    c = tqd_config()
    for f in ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "intermediate", "vocab"):
        setattr(c, f, int(getattr(model_cfg, f)))
    c.qk_norm = int(bool(model_cfg.qk_norm))
    c.weight_type = {"q8_0": TQD_WEIGHT_Q8_0, "bf16": TQD_WEIGHT_BF16}[model_cfg.weight_type]
    c.rope_theta = float(model_cfg.rope_theta)
    c.rms_eps = float(model_cfg.rms_eps)
    c.max_seq = int(max_seq)
    c.max_batch = int(max_batch)
    c.schedule = int(schedule)
    c.kv_type = int(kv_type)
    return c


class HostWeights:
    """tqd_host_weights over host arrays; keeps the arrays alive."""

    def __init__(self, layers, lm_head, out_norm, embed=None):
        self._keep = [lm_head, out_norm, embed, layers]
        n = len(layers)
        self._layers = (tqd_layer_weights * n)()
        for i, d in enumerate(layers):
            for f in _LAYER_FIELDS:
                setattr(self._layers[i], f, _ptr(d.get(f)))
        self.struct = tqd_host_weights()
        self.struct.layers = ctypes.cast(self._layers, ctypes.POINTER(tqd_layer_weights))
        self.struct.out_norm = _ptr(out_norm)
        self.struct.lm_head = _ptr(lm_head)
        self.struct.embed = _ptr(embed)


def make_host_weights(model) -> HostWeights:
    """From an object with .layers (list of dicts of arrays), .lm_head,
    .out_norm and optionally .embed."""
    return HostWeights(model.layers, model.lm_head, model.out_norm, getattr(model, "embed", None))


# ------------------------------------------------------------------ C ABI calls

def tqd_status_name(status: int) -> str:
    return lib().tqd_status_name(int(status)).decode()


def tqd_create(config: tqd_config, weights: HostWeights, stream=None) -> int:
    h = ctypes.c_void_p()
    check(lib().tqd_create(ctypes.byref(config), ctypes.byref(weights.struct), _stream(stream),
                           ctypes.byref(h)), "tqd_create")
    return h.value


def tqd_create_synthetic(config: tqd_config, seed: int, stream=None) -> int:
    h = ctypes.c_void_p()
    check(lib().tqd_create_synthetic(ctypes.byref(config), ctypes.c_uint64(seed), _stream(stream), ctypes.byref(h)),
          "tqd_create_synthetic")
    return h.value


def tqd_export_weights(handle, model_cfg) -> dict:
    """The model's weights in the upload format: {"layers": [dict name ->
    array], "lm_head": ..., "out_norm": ...} (host arrays allocated here)."""
    H, hd, I, V = model_cfg.hidden, model_cfg.head_dim, model_cfg.intermediate, model_cfg.vocab
    qw, kvw = model_cfg.n_heads * hd, model_cfg.n_kv_heads * hd

    def mat(rows, cols):
        if model_cfg.weight_type == "q8_0":
            return np.zeros((rows, cols // 32 * 34), dtype=np.uint8)
        return np.zeros((rows, cols), dtype=np.uint16)

    shapes = {"wq": (qw, H), "wk": (kvw, H), "wv": (kvw, H), "wo": (H, qw), "w_gate": (I, H), "w_up": (I, H),
              "w_down": (H, I)}
    layers = []
    for _ in range(model_cfg.n_layers):
        d = {n: mat(*shp) for n, shp in shapes.items()}
        d["attn_norm"] = np.zeros(H, dtype=np.float32)
        d["ffn_norm"] = np.zeros(H, dtype=np.float32)
        if model_cfg.qk_norm:
            d["q_norm"] = np.zeros(hd, dtype=np.float32)
            d["k_norm"] = np.zeros(hd, dtype=np.float32)
        layers.append(d)
    out = {"layers": layers, "lm_head": mat(V, H), "out_norm": np.zeros(H, dtype=np.float32)}
    hw = HostWeights(layers, out["lm_head"], out["out_norm"])
    check(lib().tqd_export_weights(handle, ctypes.byref(hw.struct)), "tqd_export_weights")
    return out


def tqd_destroy(handle) -> None:
    if handle:
        lib().tqd_destroy(handle)


def tqd_reset(handle, seq: int = 0) -> None:
    check(lib().tqd_reset(handle, seq), "tqd_reset")


def tqd_truncate(handle, seq: int, n_pos: int) -> None:
    check(lib().tqd_truncate(handle, seq, int(n_pos)), "tqd_truncate")


def tqd_next_pos(handle, seq: int = 0) -> int:
    p = ctypes.c_int32()
    check(lib().tqd_next_pos(handle, seq, ctypes.byref(p)), "tqd_next_pos")
    return p.value


def tqd_prefill(handle, seq: int, ids) -> int:
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    nxt = ctypes.c_int32()
    check(lib().tqd_prefill(handle, seq, ids.ctypes.data, ids.size, ctypes.byref(nxt)), "tqd_prefill")
    return nxt.value


def tqd_prefill_batch(handle, seq: int, ids) -> int:
    """The prompt in tiles of up to 16 positions through the batched step."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    nxt = ctypes.c_int32()
    check(lib().tqd_prefill_batch(handle, seq, ids.ctypes.data, ids.size, ctypes.byref(nxt)), "tqd_prefill_batch")
    return nxt.value


def tqd_kv_upload(handle, seq: int, k, v) -> None:
    """k, v float32 [n_layers, n_pos, kv_width] host arrays."""
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    check(lib().tqd_kv_upload(handle, seq, k.shape[1], k.ctypes.data, v.ctypes.data), "tqd_kv_upload")


def tqd_decode_step(handle, seq: int, token: int, pos: int) -> int:
    nxt = ctypes.c_int32()
    check(lib().tqd_decode_step(handle, seq, int(token), int(pos), ctypes.byref(nxt)), "tqd_decode_step")
    return nxt.value


def tqd_generate(handle, seq: int, first_token: int, n_steps: int, out=None) -> np.ndarray:
    ids = out if out is not None else np.empty(n_steps, dtype=np.int32)
    check(lib().tqd_generate(handle, seq, int(first_token), int(n_steps), ids.ctypes.data), "tqd_generate")
    return ids


def tqd_decode_step_batch(handle, tokens, pos) -> np.ndarray:
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    out = np.empty(tokens.size, dtype=np.int32)
    check(lib().tqd_decode_step_batch(handle, tokens.size, tokens.ctypes.data, pos.ctypes.data, out.ctypes.data),
          "tqd_decode_step_batch")
    return out


def tqd_generate_batch(handle, first_tokens, n_steps: int) -> np.ndarray:
    """Returns ids [n_steps, n_seq]."""
    first = np.ascontiguousarray(first_tokens, dtype=np.int32)
    out = np.empty((n_steps, first.size), dtype=np.int32)
    check(lib().tqd_generate_batch(handle, first.size, first.ctypes.data, int(n_steps), out.ctypes.data),
          "tqd_generate_batch")
    return out


def sampling(temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0, min_p: float = 0.0,
             repeat_penalty: float = 1.0, presence_penalty: float = 0.0, frequency_penalty: float = 0.0,
             seed: int = 0) -> tqd_sampling:
    """The controls of seeded sampling (neutral values switch a stage off)."""
    return tqd_sampling(temperature, top_k, top_p, min_p, repeat_penalty, presence_penalty, frequency_penalty,
                        seed & ((1 << 64) - 1))


def tqd_sample(handle, seq: int, params: tqd_sampling) -> int:
    tok = ctypes.c_int32()
    check(lib().tqd_sample(handle, seq, ctypes.byref(params), ctypes.byref(tok)), "tqd_sample")
    return tok.value


def tqd_generate_sampled(handle, seq: int, first_token: int, n_steps: int, params: tqd_sampling) -> np.ndarray:
    out = np.empty(n_steps, dtype=np.int32)
    check(lib().tqd_generate_sampled(handle, seq, first_token, n_steps, ctypes.byref(params), out.ctypes.data),
          "tqd_generate_sampled")
    return out


def tqd_generate_batch_sampled(handle, first_tokens, n_steps: int, params: tqd_sampling) -> np.ndarray:
    """Returns ids [n_steps, n_seq]."""
    first = np.ascontiguousarray(first_tokens, dtype=np.int32)
    out = np.empty((n_steps, first.size), dtype=np.int32)
    check(lib().tqd_generate_batch_sampled(handle, first.size, first.ctypes.data, int(n_steps),
                                           ctypes.byref(params), out.ctypes.data), "tqd_generate_batch_sampled")
    return out


def tqd_read_logits(handle, seq: int, vocab: int, out=None) -> np.ndarray:
    logits = out if out is not None else np.empty(vocab, dtype=np.float32)
    check(lib().tqd_read_logits(handle, seq, logits.ctypes.data), "tqd_read_logits")
    return logits


def tqd_phase_count(handle) -> int:
    n = ctypes.c_int32()
    check(lib().tqd_phase_count(handle, ctypes.byref(n)), "tqd_phase_count")
    return n.value


def tqd_step_bytes(handle, pos: int) -> int:
    b = ctypes.c_int64()
    check(lib().tqd_step_bytes(handle, int(pos), ctypes.byref(b)), "tqd_step_bytes")
    return b.value


class Decoder:
    """Owns one model handle (tqd_create ... tqd_destroy)."""

    def __init__(self, model, max_seq: int, max_batch: int = 1, schedule: int = TQD_SCHED_GRAPH,
                 stream=None, kv_type: int = TQD_KV_F32):
        self.cfg = model.cfg
        self.config = make_config(model.cfg, max_seq, max_batch, schedule, kv_type)
        self._weights = make_host_weights(model)
        self.handle = tqd_create(self.config, self._weights, stream)
        self._weights = None  # uploaded; host copies no longer needed by the library

    @classmethod
    def synthetic(cls, model_cfg, seed: int, max_seq: int, max_batch: int = 1, schedule: int = TQD_SCHED_GRAPH,
                  stream=None, kv_type: int = TQD_KV_F32):
        """A decoder over the seeded synthetic weights, generated inside the
        library (tqd_create_synthetic) rather than uploaded from host arrays."""
        self = cls.__new__(cls)
        self.cfg = model_cfg
        self.config = make_config(model_cfg, max_seq, max_batch, schedule, kv_type)
        self._weights = None
        self.handle = tqd_create_synthetic(self.config, seed, stream)
        return self

    def export_weights(self) -> dict:
        return tqd_export_weights(self.handle, self.cfg)

    def close(self):
        if getattr(self, "handle", None):
            tqd_destroy(self.handle)
            self.handle = None

    def __del__(self):
        self.close()

    def prefill(self, ids, seq: int = 0) -> int:
        return tqd_prefill(self.handle, seq, ids)

    def prefill_batch(self, ids, seq: int = 0) -> int:
        return tqd_prefill_batch(self.handle, seq, ids)

    def decode_step(self, token: int, pos: int, seq: int = 0) -> int:
        return tqd_decode_step(self.handle, seq, token, pos)

    def generate(self, first_token: int, n_steps: int, seq: int = 0) -> np.ndarray:
        return tqd_generate(self.handle, seq, first_token, n_steps)

    def decode_step_batch(self, tokens, pos) -> np.ndarray:
        return tqd_decode_step_batch(self.handle, tokens, pos)

    def generate_batch(self, first_tokens, n_steps: int) -> np.ndarray:
        return tqd_generate_batch(self.handle, first_tokens, n_steps)

    def sample(self, params: tqd_sampling, seq: int = 0) -> int:
        return tqd_sample(self.handle, seq, params)

    def generate_sampled(self, first_token: int, n_steps: int, params: tqd_sampling, seq: int = 0) -> np.ndarray:
        return tqd_generate_sampled(self.handle, seq, first_token, n_steps, params)

    def generate_batch_sampled(self, first_tokens, n_steps: int, params: tqd_sampling) -> np.ndarray:
        return tqd_generate_batch_sampled(self.handle, first_tokens, n_steps, params)

    def logits(self, seq: int = 0) -> np.ndarray:
        return tqd_read_logits(self.handle, seq, self.cfg.vocab)

    def kv_upload(self, k, v, seq: int = 0):
        tqd_kv_upload(self.handle, seq, k, v)

    def truncate(self, n_pos: int, seq: int = 0):
        tqd_truncate(self.handle, seq, n_pos)

    def next_pos(self, seq: int = 0) -> int:
        return tqd_next_pos(self.handle, seq)

    def reset(self, seq: int = 0):
        tqd_reset(self.handle, seq)

    @property
    def phase_count(self) -> int:
        return tqd_phase_count(self.handle)

    def step_bytes(self, pos: int) -> int:
        return tqd_step_bytes(self.handle, pos)


from . import ops  # noqa: E402,F401  (operator entry points on torch tensors)
