"""ORACLE — test infrastructure only.

ctypes binding of ``tqd_oracle.c``, the plain double-precision CPU restatement
of the Q8_0 greedy-decode step.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg use it; the decode library never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tqd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libtqd_oracle.so")

Q8_0, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc: -O2, OpenMP, IEEE semantics (no fast-math,
    no FMA contraction), so x86-64 and aarch64 hosts produce the same bits."""
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
        vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.orc_f16_to_f64.restype = dbl
        L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f64.restype = dbl
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_q8_0_dequant_block.restype = None
        L.orc_q8_0_dequant_block.argtypes = [vp, vp]
        L.orc_q8_0_matvec.restype = None
        L.orc_q8_0_matvec.argtypes = [vp, i64, i64, vp, vp]
        L.orc_bf16_matvec.restype = None
        L.orc_bf16_matvec.argtypes = [vp, i64, i64, vp, vp]
        L.orc_rmsnorm.restype = None
        L.orc_rmsnorm.argtypes = [vp, vp, i64, dbl, vp]
        L.orc_rmsnorm_rows.restype = None
        L.orc_rmsnorm_rows.argtypes = [vp, vp, i64, i64, dbl, vp]
        L.orc_rope.restype = None
        L.orc_rope.argtypes = [vp, i32, i32, i64, dbl]
        L.orc_attention.restype = None
        L.orc_attention.argtypes = [vp, vp, vp, i64, i64, i32, i32, i32, vp]
        L.orc_silu.restype = dbl
        L.orc_silu.argtypes = [dbl]
        L.orc_silu_mul.restype = None
        L.orc_silu_mul.argtypes = [vp, vp, i64, vp]
        L.orc_argmax.restype = i64
        L.orc_argmax.argtypes = [vp, i64]
        L.orc_model_new.restype = vp
        L.orc_model_new.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, dbl, dbl, i64]
        L.orc_model_free.restype = None
        L.orc_model_free.argtypes = [vp]
        L.orc_model_set_layer.restype = i32
        L.orc_model_set_layer.argtypes = [vp, i32] + [vp] * 11
        L.orc_model_set_head.restype = i32
        L.orc_model_set_head.argtypes = [vp, vp, vp, vp]
        L.orc_step.restype = i32
        L.orc_step.argtypes = [vp, i64, i64, i32, vp, ctypes.POINTER(i64)]
        L.orc_get_hidden.restype = None
        L.orc_get_hidden.argtypes = [vp, vp]
        L.orc_kv_get.restype = i32
        L.orc_kv_get.argtypes = [vp, i32, i64, vp, vp]
        L.orc_kv_load.restype = i32
        L.orc_kv_load.argtypes = [vp, i64, vp, vp]
        L.orc_set_kv_f16.restype = i32
        L.orc_set_kv_f16.argtypes = [vp, i32]
        L.orc_next_pos.restype = i64
        L.orc_next_pos.argtypes = [vp]
        L.orc_reset.restype = None
        L.orc_reset.argtypes = [vp]
        L.orc_max_threads.restype = i32
        L.orc_max_threads.argtypes = []
        L.orc_set_threads.restype = None
        L.orc_set_threads.argtypes = [i32]
        _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


# ---------------------------------------------------------------- per-op functions

def f16_to_f64(bits: int) -> float:
    return lib().orc_f16_to_f64(int(bits))


def bf16_to_f64(bits: int) -> float:
    return lib().orc_bf16_to_f64(int(bits))


def q8_0_dequant_block(blk: np.ndarray) -> np.ndarray:
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    out = np.empty(32, dtype=np.float64)
    lib().orc_q8_0_dequant_block(_p(blk), _p(out))
    return out


def q8_0_matvec(w: np.ndarray, cols: int, x) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.uint8)
    rows = w.size // (cols // 32 * 34)
    x = _f64(x)
    y = np.empty(rows, dtype=np.float64)
    lib().orc_q8_0_matvec(_p(w), rows, cols, _p(x), _p(y))
    return y


def bf16_matvec(w: np.ndarray, x) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.uint16)
    rows, cols = w.shape
    x = _f64(x)
    y = np.empty(rows, dtype=np.float64)
    lib().orc_bf16_matvec(_p(w), rows, cols, _p(x), _p(y))
    return y


def rmsnorm(x, g, eps: float) -> np.ndarray:
    x = _f64(x)
    g = _f32(g)
    n = g.size
    rows = x.size // n
    out = np.empty_like(x)
    lib().orc_rmsnorm_rows(_p(x), _p(g), rows, n, eps, _p(out))
    return out


def rope(x, n_heads: int, head_dim: int, pos: int, theta: float) -> np.ndarray:
    x = _f64(x).copy()
    lib().orc_rope(_p(x), n_heads, head_dim, pos, theta)
    return x


def attention(q, K, V, n_heads: int, n_kv: int, head_dim: int) -> np.ndarray:
    """q [n_heads*hd]; K, V [S, n_kv*hd] -> [n_heads*hd]."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    S = K.shape[0]
    out = np.empty(n_heads * head_dim, dtype=np.float64)
    lib().orc_attention(_p(q), _p(K), _p(V), S, n_kv * head_dim, n_heads, n_kv, head_dim, _p(out))
    return out


def silu(z: float) -> float:
    return lib().orc_silu(float(z))


def silu_mul(g, u) -> np.ndarray:
    g, u = _f64(g), _f64(u)
    out = np.empty_like(g)
    lib().orc_silu_mul(_p(g), _p(u), g.size, _p(out))
    return out


def argmax(x) -> int:
    x = _f64(x)
    return int(lib().orc_argmax(_p(x), x.size))


def max_threads() -> int:
    return int(lib().orc_max_threads())


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


# ---------------------------------------------------------------- the model

class OracleModel:
    """One sequence of the reference decoder over a synthetic model's arrays.

    ``model`` is a ``synth.SynthModel`` (or any object with the same fields);
    its arrays are referenced, not copied, so they must outlive this object."""

    def __init__(self, model, max_seq: int, kv_f16: bool = False):
        cfg = model.cfg
        self.cfg = cfg
        self._model = model
        wt = Q8_0 if cfg.weight_type == "q8_0" else BF16
        L = lib()
        self._h = L.orc_model_new(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim,
                                  cfg.intermediate, cfg.vocab, int(cfg.qk_norm), wt,
                                  cfg.rope_theta, cfg.rms_eps, max_seq)
        if not self._h:
            raise ValueError("oracle rejected the configuration")
        for l, d in enumerate(model.layers):
            rc = L.orc_model_set_layer(self._h, l, _p(d["attn_norm"]), _p(d["wq"]), _p(d["wk"]),
                                       _p(d["wv"]), _p(d["wo"]), _p(d.get("q_norm")),
                                       _p(d.get("k_norm")), _p(d["ffn_norm"]), _p(d["w_gate"]),
                                       _p(d["w_up"]), _p(d["w_down"]))
            assert rc == 0
        assert L.orc_model_set_head(self._h, _p(model.lm_head), _p(model.out_norm), None) == 0
        assert L.orc_set_kv_f16(self._h, int(kv_f16)) == 0
        self.max_seq = max_seq

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().orc_model_free(h)
            self._h = None

    def step(self, token: int, pos: int, want_logits: bool = True):
        """Run one step; returns (next_id, logits f64[vocab]) or (-1, None)."""
        logits = np.empty(self.cfg.vocab, dtype=np.float64) if want_logits else None
        nxt = ctypes.c_int64(-1)
        rc = lib().orc_step(self._h, int(token), int(pos), int(want_logits), _p(logits), ctypes.byref(nxt))
        if rc == -1:
            raise ValueError("oracle step: bad token or position")
        if rc == -2:
            raise FloatingPointError("oracle step: every logit is NaN")
        return int(nxt.value), logits

    def prefill(self, ids, start: int = 0):
        """Steps over ids at positions start.. ; logits only at the last one."""
        ids = list(int(t) for t in ids)
        for i, t in enumerate(ids[:-1]):
            self.step(t, start + i, want_logits=False)
        return self.step(ids[-1], start + len(ids) - 1, want_logits=True)

    def hidden(self) -> np.ndarray:
        out = np.empty(self.cfg.hidden, dtype=np.float64)
        lib().orc_get_hidden(self._h, _p(out))
        return out

    def kv_row(self, layer: int, pos: int):
        kvw = self.cfg.kv_width
        k = np.empty(kvw, dtype=np.float64)
        v = np.empty(kvw, dtype=np.float64)
        assert lib().orc_kv_get(self._h, layer, pos, _p(k), _p(v)) == 0
        return k, v

    def kv_load(self, k: np.ndarray, v: np.ndarray):
        """k, v float32 [n_layers, n_pos, kv_width]; sets the next position to n_pos."""
        k, v = _f32(k), _f32(v)
        n_pos = k.shape[1]
        assert lib().orc_kv_load(self._h, n_pos, _p(k), _p(v)) == 0

    @property
    def next_pos(self) -> int:
        return int(lib().orc_next_pos(self._h))

    def reset(self):
        lib().orc_reset(self._h)
