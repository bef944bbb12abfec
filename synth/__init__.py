"""Seeded synthetic inputs shared by the oracle and the CUDA library.

The arithmetic that defines each draw lives in ``tqd_synth.c`` (see its header);
this module compiles it, exposes it through ctypes, and assembles whole models,
prompts and KV fills for the five named workloads.  It holds none of the decode
step's arithmetic: everything here is input construction, consumed byte for byte
by both sides.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tqd_synth.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libtqd_synth.so")

# Tensor stream indices: the tied embedding / lm_head matrix is 0, layer l's
# tensors follow in the order below, the final norm comes last.
LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "q_norm", "k_norm",
                 "ffn_norm", "w_gate", "w_up", "w_down")
PROMPT_STREAM_BASE = 0x10000
KV_FILL_STREAM_BASE = 0x20000


def build(force: bool = False) -> str:
    """Compile the generator with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
        vp = ctypes.c_void_p
        L.tqs_stream.restype = u64
        L.tqs_stream.argtypes = [u64, u64]
        L.tqs_draw.restype = u64
        L.tqs_draw.argtypes = [u64, u64]
        L.tqs_std_normal.restype = dbl
        L.tqs_std_normal.argtypes = [u64, u64]
        L.tqs_f32_to_f16.restype = ctypes.c_uint16
        L.tqs_f32_to_f16.argtypes = [ctypes.c_float]
        L.tqs_f32_to_bf16.restype = ctypes.c_uint16
        L.tqs_f32_to_bf16.argtypes = [ctypes.c_float]
        L.tqs_normal_f32.restype = None
        L.tqs_normal_f32.argtypes = [u64, u64, i64, dbl, dbl, vp]
        L.tqs_quantize_block.restype = None
        L.tqs_quantize_block.argtypes = [vp, vp]
        L.tqs_q8_0_matrix.restype = ctypes.c_int
        L.tqs_q8_0_matrix.argtypes = [u64, u64, i64, i64, dbl, vp]
        L.tqs_bf16_matrix.restype = ctypes.c_int
        L.tqs_bf16_matrix.argtypes = [u64, u64, i64, i64, dbl, vp]
        L.tqs_token_ids.restype = None
        L.tqs_token_ids.argtypes = [u64, i64, i64, i64, vp]
        L.tqs_uniform_f32.restype = None
        L.tqs_uniform_f32.argtypes = [u64, u64, i64, dbl, dbl, vp]
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------
# primitive draws
# --------------------------------------------------------------------------

def normal_f32(seed: int, tensor: int, n: int, mean: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().tqs_normal_f32(seed, tensor, n, mean, sigma, _ptr(out))
    return out


def uniform_f32(seed: int, tensor: int, n: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().tqs_uniform_f32(seed, tensor, n, lo, hi, _ptr(out))
    return out


def q8_0_matrix(seed: int, tensor: int, rows: int, cols: int, sigma: float = 0.02) -> np.ndarray:
    """Q8_0 bytes of a [rows x cols] N(0, sigma) matrix: uint8 [rows, cols/32*34]."""
    if cols % 32:
        raise ValueError("Q8_0 needs cols % 32 == 0")
    out = np.empty((rows, cols // 32 * 34), dtype=np.uint8)
    rc = lib().tqs_q8_0_matrix(seed, tensor, rows, cols, sigma, _ptr(out))
    assert rc == 0
    return out


def bf16_matrix(seed: int, tensor: int, rows: int, cols: int, sigma: float = 0.02) -> np.ndarray:
    """bf16 bit patterns (uint16 [rows, cols]) of a N(0, sigma) matrix."""
    out = np.empty((rows, cols), dtype=np.uint16)
    rc = lib().tqs_bf16_matrix(seed, tensor, rows, cols, sigma, _ptr(out))
    assert rc == 0
    return out


def quantize_rows(w: np.ndarray) -> np.ndarray:
    """Q8_0-encode an arbitrary f32 matrix [rows, cols] (cols % 32 == 0)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    if cols % 32:
        raise ValueError("Q8_0 needs cols % 32 == 0")
    out = np.empty((rows, cols // 32 * 34), dtype=np.uint8)
    L = lib()
    flat = w.reshape(-1, 32)
    ob = out.reshape(-1, 34)
    for i in range(flat.shape[0]):
        L.tqs_quantize_block(flat[i].ctypes.data_as(ctypes.c_void_p), ob[i].ctypes.data_as(ctypes.c_void_p))
    return out


def f32_to_f16_bits(x: float) -> int:
    return int(lib().tqs_f32_to_f16(float(x)))


def f32_to_bf16_bits(x: float) -> int:
    return int(lib().tqs_f32_to_bf16(float(x)))


def token_ids(seed: int, seq: int, n: int, vocab: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    lib().tqs_token_ids(seed, seq, n, vocab, _ptr(out))
    return out


# --------------------------------------------------------------------------
# model configurations and whole synthetic models
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class ModelConfig:
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    qk_norm: bool
    weight_type: str  # "q8_0" or "bf16"
    rope_theta: float
    rms_eps: float = 1e-6

    @property
    def q_width(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.n_kv_heads * self.head_dim


@dataclass(frozen=True)
class Workload:
    name: str
    model: ModelConfig
    prompt_len: int
    decode_steps: int
    batch: int = 1
    model_seed: int = 0
    prompt_seed: int = 1000


QWEN3_06B = ModelConfig(28, 1024, 16, 8, 128, 3072, 151936, True, "q8_0", 1e6)
SMOLLM2_360M = ModelConfig(32, 960, 15, 5, 64, 2560, 49152, False, "bf16", 1e5)
TINY = ModelConfig(2, 256, 4, 2, 64, 768, 4096, True, "q8_0", 1e6)

WORKLOADS = {
    "tiny": Workload("tiny-qwen3-2L-h256-q8_0", TINY, 32, 16),
    "qwen3_0.6b": Workload("qwen3-0.6b-shape-q8_0-prompt511-decode128", QWEN3_06B, 511, 128),
    "smollm2_360m": Workload("smollm2-360m-shape-bf16-prompt256-decode128", SMOLLM2_360M, 256, 128),
    "qwen3_0.6b_long": Workload("qwen3-0.6b-shape-q8_0-kv4096-decode64", QWEN3_06B, 4096, 64),
    "qwen3_0.6b_batch16": Workload("qwen3-0.6b-shape-q8_0-16x1024-decode64", QWEN3_06B, 1024, 64, batch=16),
    "qwen3_0.6b_batch32": Workload("qwen3-0.6b-shape-q8_0-32x1024-decode64", QWEN3_06B, 1024, 64, batch=32),
}


def layer_tensor_index(layer: int, name: str) -> int:
    return 1 + 11 * layer + LAYER_TENSORS.index(name)


def out_norm_index(cfg: ModelConfig) -> int:
    return 1 + 11 * cfg.n_layers


@dataclass
class SynthModel:
    """Host copies of every weight tensor, in the decoder's on-disk formats.

    Matrices are Q8_0 bytes ([rows, cols/32*34] uint8) or bf16 bit patterns
    ([rows, cols] uint16); norm gains are float32.  ``lm_head`` doubles as the
    token embedding (tied weights)."""
    cfg: ModelConfig
    seed: int
    lm_head: np.ndarray
    out_norm: np.ndarray
    layers: list = field(default_factory=list)  # list of dict name -> array


def make_matrix(cfg: ModelConfig, seed: int, tensor: int, rows: int, cols: int, sigma: float = 0.02):
    if cfg.weight_type == "q8_0":
        return q8_0_matrix(seed, tensor, rows, cols, sigma)
    if cfg.weight_type == "bf16":
        return bf16_matrix(seed, tensor, rows, cols, sigma)
    raise ValueError(cfg.weight_type)


def make_model(cfg: ModelConfig, seed: int = 0, zero_matrices: tuple = ()) -> SynthModel:
    """Weights ~N(0, 0.02) (Q8_0 or bf16), gains 1 + N(0, 0.1) in f32.

    ``zero_matrices`` names layer matrices to replace by all-zero blocks (the
    special cases that reduce the step to closed forms)."""
    H, qw, kvw, I, hd = cfg.hidden, cfg.q_width, cfg.kv_width, cfg.intermediate, cfg.head_dim
    shapes = {"wq": (qw, H), "wk": (kvw, H), "wv": (kvw, H), "wo": (H, qw),
              "w_gate": (I, H), "w_up": (I, H), "w_down": (H, I)}
    gains = {"attn_norm": H, "q_norm": hd, "k_norm": hd, "ffn_norm": H}
    lm = make_matrix(cfg, seed, 0, cfg.vocab, H)
    layers = []
    for l in range(cfg.n_layers):
        d = {}
        for name in LAYER_TENSORS:
            t = layer_tensor_index(l, name)
            if name in shapes:
                r, c = shapes[name]
                if name in zero_matrices:
                    if cfg.weight_type == "q8_0":
                        d[name] = np.zeros((r, c // 32 * 34), dtype=np.uint8)
                    else:
                        d[name] = np.zeros((r, c), dtype=np.uint16)
                else:
                    d[name] = make_matrix(cfg, seed, t, r, c)
            else:
                if name in ("q_norm", "k_norm") and not cfg.qk_norm:
                    continue
                d[name] = normal_f32(seed, t, gains[name], 1.0, 0.1)
        layers.append(d)
    on = normal_f32(seed, out_norm_index(cfg), H, 1.0, 0.1)
    return SynthModel(cfg, seed, lm, on, layers)


def prompt(wl: Workload, seq: int = 0) -> np.ndarray:
    return token_ids(wl.prompt_seed, seq, wl.prompt_len, wl.model.vocab)


def kv_fill(cfg: ModelConfig, seed: int, seq: int, n_pos: int, lo: float = -1.0, hi: float = 1.0):
    """A seeded stand-in KV history: K and V f32 [n_layers, n_pos, kv_width]."""
    n = cfg.n_layers * n_pos * cfg.kv_width
    k = uniform_f32(seed, KV_FILL_STREAM_BASE + 2 * seq, n, lo, hi)
    v = uniform_f32(seed, KV_FILL_STREAM_BASE + 2 * seq + 1, n, lo, hi)
    shape = (cfg.n_layers, n_pos, cfg.kv_width)
    return k.reshape(shape), v.reshape(shape)
