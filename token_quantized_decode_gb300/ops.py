"""Operator entry points of libtqd on torch CUDA tensors (tqd_op_* in
include/tqd.h).  Each call marshals data pointers and the current stream into
one C call; outputs are written into caller-allocated tensors."""
from __future__ import annotations

from ._lib import check, lib


def _s(stream):
    import torch
    return int((stream or torch.cuda.current_stream()).cuda_stream)


def tqd_op_q8_0_repack(w_blocks, rows: int, cols: int, w_rows, stream=None):
    check(lib().tqd_op_q8_0_repack(w_blocks.data_ptr(), rows, cols, w_rows.data_ptr(), _s(stream)),
          "tqd_op_q8_0_repack")


def tqd_op_q8_0_matvec(w_rows, rows: int, cols: int, x, y, stream=None):
    check(lib().tqd_op_q8_0_matvec(w_rows.data_ptr(), rows, cols, x.data_ptr(), y.data_ptr(), _s(stream)),
          "tqd_op_q8_0_matvec")


def tqd_op_bf16_matvec(w, rows: int, cols: int, x, y, stream=None):
    check(lib().tqd_op_bf16_matvec(w.data_ptr(), rows, cols, x.data_ptr(), y.data_ptr(), _s(stream)),
          "tqd_op_bf16_matvec")


def tqd_op_rmsnorm(x, g, rows: int, n: int, eps: float, out, stream=None):
    check(lib().tqd_op_rmsnorm(x.data_ptr(), g.data_ptr(), rows, n, eps, out.data_ptr(), _s(stream)),
          "tqd_op_rmsnorm")


def tqd_op_rope_table(theta: float, head_dim: int, max_pos: int, table, stream=None):
    check(lib().tqd_op_rope_table(theta, head_dim, max_pos, table.data_ptr(), _s(stream)), "tqd_op_rope_table")


def tqd_op_rope(x, n_heads: int, head_dim: int, pos: int, table, stream=None):
    check(lib().tqd_op_rope(x.data_ptr(), n_heads, head_dim, pos, table.data_ptr(), _s(stream)), "tqd_op_rope")


def tqd_attention_scratch_bytes(n_heads: int, n_kv: int, head_dim: int, n_chunks: int) -> int:
    return int(lib().tqd_attention_scratch_bytes(n_heads, n_kv, head_dim, n_chunks))


def tqd_op_attention(q, K, V, S: int, n_heads: int, n_kv: int, head_dim: int, n_chunks: int, out,
                     scratch, stream=None):
    check(lib().tqd_op_attention(q.data_ptr(), K.data_ptr(), V.data_ptr(), S, n_heads, n_kv, head_dim,
                                 n_chunks, out.data_ptr(), scratch.data_ptr(), _s(stream)),
          "tqd_op_attention")


def tqd_op_attention_noalloc(q, K, V, S: int, n_heads: int, n_kv: int, head_dim: int, n_chunks: int, out,
                             stream=None):
    """tqd_op_attention without caller scratch: the library's static device
    array holds the partials (allocates nothing per call)."""
    check(lib().tqd_op_attention_noalloc(q.data_ptr(), K.data_ptr(), V.data_ptr(), S, n_heads, n_kv, head_dim,
                                         n_chunks, out.data_ptr(), _s(stream)),
          "tqd_op_attention_noalloc")


def tqd_op_attention_noalloc_max_scratch() -> int:
    return int(lib().tqd_op_attention_noalloc_max_scratch())


def tqd_op_wait_selftest(stream=None):
    """Run the bounded-wait self-test; returns (status, error bits) without
    raising (the expected status is TQD_ERR_DEVICE_TIMEOUT)."""
    import ctypes
    bits = ctypes.c_uint32(0)
    status = lib().tqd_op_wait_selftest(_s(stream), ctypes.byref(bits))
    return int(status), int(bits.value)


def tqd_op_silu_mul(g, u, n: int, out, stream=None):
    check(lib().tqd_op_silu_mul(g.data_ptr(), u.data_ptr(), n, out.data_ptr(), _s(stream)), "tqd_op_silu_mul")


def tqd_argmax_scratch_bytes() -> int:
    return int(lib().tqd_argmax_scratch_bytes())


def tqd_op_argmax(x, n: int, idx_out, scratch, stream=None):
    check(lib().tqd_op_argmax(x.data_ptr(), n, idx_out.data_ptr(), scratch.data_ptr(), _s(stream)),
          "tqd_op_argmax")


def tqd_sample_scratch_bytes(vocab: int) -> int:
    return int(lib().tqd_sample_scratch_bytes(vocab))


def tqd_op_sample(logits, vocab: int, tokens, n_inputs: int, params, scratch, stream=None):
    """The seeded draw of tqd_sample on caller tensors: tokens[:n_inputs] are
    the inputs so far, the drawn token is written to tokens[n_inputs]."""
    import ctypes
    check(lib().tqd_op_sample(logits.data_ptr(), vocab, tokens.data_ptr(), n_inputs, ctypes.byref(params),
                              scratch.data_ptr(), _s(stream)),
          "tqd_op_sample")
