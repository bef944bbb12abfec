"""ctypes declarations of libtqd's C ABI (include/tqd.h).

Loading fails loudly when the compiled library is missing: there is no
fallback implementation of anything in this package.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtqd.so")

TQD_OK = 0
STATUS_NAMES = [
    "TQD_OK", "TQD_ERR_BAD_ARG", "TQD_ERR_UNSUPPORTED_CONFIG", "TQD_ERR_NO_DEVICE", "TQD_ERR_CUDA",
    "TQD_ERR_OOM", "TQD_ERR_CAPACITY", "TQD_ERR_POS_MISMATCH", "TQD_ERR_DEVICE_TIMEOUT",
    "TQD_ERR_NUMERIC", "TQD_ERR_POISONED", "TQD_ERR_NOT_PREFILLED",
]
for _i, _n in enumerate(STATUS_NAMES):
    globals()[_n] = _i

TQD_WEIGHT_Q8_0, TQD_WEIGHT_BF16 = 0, 1
TQD_SCHED_GRAPH, TQD_SCHED_PERSISTENT = 0, 1
TQD_KV_F32, TQD_KV_F16 = 0, 1


class tqd_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("intermediate", ctypes.c_int32), ("vocab", ctypes.c_int32), ("qk_norm", ctypes.c_int32),
                ("weight_type", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("max_seq", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("schedule", ctypes.c_int32), ("kv_type", ctypes.c_int32)]


class tqd_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "wq", "wk", "wv", "wo", "q_norm", "k_norm",
                                               "ffn_norm", "w_gate", "w_up", "w_down")]


class tqd_host_weights(ctypes.Structure):
    _fields_ = [("layers", ctypes.POINTER(tqd_layer_weights)), ("out_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p), ("embed", ctypes.c_void_p)]


class tqd_sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float),
                ("min_p", ctypes.c_float), ("repeat_penalty", ctypes.c_float),
                ("presence_penalty", ctypes.c_float), ("frequency_penalty", ctypes.c_float),
                ("seed", ctypes.c_uint64)]


class TQDError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        self.name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else f"status {status}"
        super().__init__(f"{where}: {self.name}" + (f" ({detail})" if detail else ""))


_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libtqd is not built ({LIB_PATH} missing); run __graft_entry__.build() "
                          "or python token_quantized_decode_gb300/build.py")
    L = ctypes.CDLL(LIB_PATH)
    i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "tqd_status_name": (ctypes.c_char_p, [i32]),
        "tqd_last_error": (ctypes.c_char_p, []),
        "tqd_create": (i32, [P(tqd_config), P(tqd_host_weights), vp, P(vp)]),
        "tqd_create_synthetic": (i32, [P(tqd_config), ctypes.c_uint64, vp, P(vp)]),
        "tqd_export_weights": (i32, [vp, P(tqd_host_weights)]),
        "tqd_destroy": (None, [vp]),
        "tqd_reset": (i32, [vp, i32]),
        "tqd_truncate": (i32, [vp, i32, i32]),
        "tqd_next_pos": (i32, [vp, i32, P(i32)]),
        "tqd_prefill": (i32, [vp, i32, vp, i32, P(i32)]),
        "tqd_prefill_batch": (i32, [vp, i32, vp, i32, P(i32)]),
        "tqd_kv_upload": (i32, [vp, i32, i32, vp, vp]),
        "tqd_decode_step": (i32, [vp, i32, i32, i32, P(i32)]),
        "tqd_generate": (i32, [vp, i32, i32, i32, vp]),
        "tqd_decode_step_batch": (i32, [vp, i32, vp, vp, vp]),
        "tqd_generate_batch": (i32, [vp, i32, vp, i32, vp]),
        "tqd_sample": (i32, [vp, i32, P(tqd_sampling), P(i32)]),
        "tqd_generate_sampled": (i32, [vp, i32, i32, i32, P(tqd_sampling), vp]),
        "tqd_generate_batch_sampled": (i32, [vp, i32, vp, i32, P(tqd_sampling), vp]),
        "tqd_read_logits": (i32, [vp, i32, vp]),
        "tqd_phase_count": (i32, [vp, P(i32)]),
        "tqd_step_bytes": (i32, [vp, i32, P(i64)]),
        "tqd_op_q8_0_repack": (i32, [vp, i64, i64, vp, vp]),
        "tqd_op_q8_0_matvec": (i32, [vp, i64, i64, vp, vp, vp]),
        "tqd_op_bf16_matvec": (i32, [vp, i64, i64, vp, vp, vp]),
        "tqd_op_rmsnorm": (i32, [vp, vp, i32, i32, ctypes.c_float, vp, vp]),
        "tqd_op_rope_table": (i32, [ctypes.c_float, i32, i32, vp, vp]),
        "tqd_op_rope": (i32, [vp, i32, i32, i32, vp, vp]),
        "tqd_op_attention": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]),
        "tqd_attention_scratch_bytes": (sz, [i32, i32, i32, i32]),
        "tqd_op_wait_selftest": (i32, [vp, P(ctypes.c_uint32)]),
        "tqd_op_silu_mul": (i32, [vp, vp, i64, vp, vp]),
        "tqd_op_argmax": (i32, [vp, i64, vp, vp, vp]),
        "tqd_argmax_scratch_bytes": (sz, []),
        "tqd_op_sample": (i32, [vp, i32, vp, i32, P(tqd_sampling), vp, vp]),
        "tqd_sample_scratch_bytes": (sz, [i32]),
        "tqd_op_attention_noalloc": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]),
        "tqd_op_attention_noalloc_max_scratch": (sz, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def exported_symbols():
    """Names the C ABI declares, in header order."""
    return [
        "tqd_create_synthetic", "tqd_export_weights", "tqd_status_name", "tqd_last_error", "tqd_create", "tqd_destroy", "tqd_reset", "tqd_truncate", "tqd_next_pos",
        "tqd_prefill", "tqd_prefill_batch", "tqd_kv_upload", "tqd_decode_step", "tqd_generate", "tqd_decode_step_batch",
        "tqd_generate_batch", "tqd_sample", "tqd_generate_sampled", "tqd_generate_batch_sampled",
        "tqd_read_logits",
        "tqd_phase_count", "tqd_step_bytes", "tqd_op_q8_0_repack", "tqd_op_q8_0_matvec",
        "tqd_op_bf16_matvec", "tqd_op_rmsnorm", "tqd_op_rope_table", "tqd_op_rope", "tqd_op_attention",
        "tqd_attention_scratch_bytes", "tqd_op_wait_selftest", "tqd_op_silu_mul", "tqd_op_argmax", "tqd_argmax_scratch_bytes",
        "tqd_op_sample", "tqd_sample_scratch_bytes", "tqd_op_attention_noalloc", "tqd_op_attention_noalloc_max_scratch",
    ]


def check(status: int, where: str):
    if status != TQD_OK:
        detail = lib().tqd_last_error().decode(errors="replace")
        raise TQDError(status, where, detail)
