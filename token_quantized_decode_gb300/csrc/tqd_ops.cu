// Operator entry points of libtqd: each runs one phase of the decode step on
// caller-owned device memory (contracts in tqd.h).  They exist so that every
// piece can be checked on its own, as in the inferno.rs blog's "The
// correctness ladder", rung one.
#include <cuda_runtime.h>

#include "tqd.h"
#include "tqd_internal.h"

using namespace tqd;

namespace {

int32_t status_of(cudaError_t e) {
  if (e == cudaSuccess) return TQD_OK;
  if (e == cudaErrorInvalidValue) return TQD_ERR_BAD_ARG;
  return TQD_ERR_CUDA;
}

size_t attn_scratch_floats_o(int32_t nq, int32_t hd, int32_t nch) {
  return static_cast<size_t>(nq) * nch * hd;
}
size_t attn_scratch_floats_ml(int32_t nq, int32_t nch) { return static_cast<size_t>(nq) * nch * 2; }

}  // namespace

extern "C" {

int32_t tqd_op_q8_0_repack(const uint8_t* w_blocks, int64_t rows, int64_t cols, uint8_t* w_rows,
                           void* stream) {
  if (!w_blocks || !w_rows || rows <= 0 || cols <= 0 || cols % 32) return TQD_ERR_BAD_ARG;
  return status_of(
      launch_q8_repack(w_blocks, rows, cols, w_rows, 0, 1, static_cast<cudaStream_t>(stream)));
}

int32_t tqd_op_q8_0_matvec(const uint8_t* w_rows, int64_t rows, int64_t cols, const float* x,
                           float* y, void* stream) {
  if (!w_rows || !x || !y || rows <= 0 || rows > (1ll << 30) || cols <= 0 || cols % 32 ||
      matvec_cpl(0, static_cast<int>(cols)) == 0)
    return TQD_ERR_BAD_ARG;
  return status_of(launch_op_matvec(0, w_rows, q8_row_bytes(cols),
                                    static_cast<int>(rows), static_cast<int>(cols), x, y,
                                    static_cast<cudaStream_t>(stream)));
}

int32_t tqd_op_bf16_matvec(const uint16_t* w, int64_t rows, int64_t cols, const float* x, float* y,
                           void* stream) {
  if (!w || !x || !y || rows <= 0 || rows > (1ll << 30) || cols <= 0 || cols % 8 ||
      matvec_cpl(1, static_cast<int>(cols)) == 0)
    return TQD_ERR_BAD_ARG;
  return status_of(launch_op_matvec(1, reinterpret_cast<const uint8_t*>(w),
                                    static_cast<size_t>(cols) * 2, static_cast<int>(rows),
                                    static_cast<int>(cols), x, y,
                                    static_cast<cudaStream_t>(stream)));
}

int32_t tqd_op_rmsnorm(const float* x, const float* g, int32_t rows, int32_t n, float eps,
                       float* out, void* stream) {
  if (!x || !g || !out || rows <= 0 || n <= 0 || n > 12 * 1024 || rows > 65535)
    return TQD_ERR_BAD_ARG;
  return status_of(launch_op_rmsnorm(x, g, rows, n, eps, out, static_cast<cudaStream_t>(stream)));
}

int32_t tqd_op_rope_table(float theta, int32_t head_dim, int32_t max_pos, float* table,
                          void* stream) {
  if (!table || !(theta > 0.f) || head_dim <= 0 || head_dim % 2 || max_pos <= 0)
    return TQD_ERR_BAD_ARG;
  return status_of(launch_rope_table(static_cast<double>(theta), head_dim, max_pos,
                                     reinterpret_cast<float2*>(table),
                                     static_cast<cudaStream_t>(stream)));
}

int32_t tqd_op_rope(float* x, int32_t n_heads, int32_t head_dim, int32_t pos, const float* table,
                    void* stream) {
  if (!x || !table || n_heads <= 0 || pos < 0 || (head_dim != 64 && head_dim != 128))
    return TQD_ERR_BAD_ARG;
  const float2* row = reinterpret_cast<const float2*>(table) + static_cast<size_t>(pos) * (head_dim / 2);
  return status_of(launch_op_rope(x, n_heads, head_dim, row, static_cast<cudaStream_t>(stream)));
}

size_t tqd_attention_scratch_bytes(int32_t n_heads, int32_t n_kv, int32_t head_dim,
                                   int32_t n_chunks) {
  if (n_heads <= 0 || n_kv <= 0 || head_dim <= 0 || n_chunks <= 0) return 0;
  const size_t o = attn_scratch_floats_o(n_heads, head_dim, n_chunks) * 4;
  const size_t ml = attn_scratch_floats_ml(n_heads, n_chunks) * 4;
  return o + ml + static_cast<size_t>(n_kv) * 4;
}

int32_t tqd_op_attention(const float* q, const float* K, const float* V, int32_t S,
                         int32_t n_heads, int32_t n_kv, int32_t head_dim, int32_t n_chunks,
                         float* out, void* scratch, void* stream) {
  if (!q || !K || !V || !out || !scratch || S <= 0 || n_heads <= 0 || n_kv <= 0 ||
      n_heads % n_kv || n_chunks < 1 || n_chunks > 1024 || n_kv * n_chunks > (1 << 20) ||
      !attention_supported(head_dim, n_heads / n_kv))
    return TQD_ERR_BAD_ARG;
  float* po = static_cast<float*>(scratch);
  float* pml = po + attn_scratch_floats_o(n_heads, head_dim, n_chunks);
  uint32_t* cnt =
      reinterpret_cast<uint32_t*>(pml + attn_scratch_floats_ml(n_heads, n_chunks));
  return status_of(launch_op_attention(q, K, V, S, n_heads, n_kv, head_dim, n_chunks, out, po, pml,
                                       cnt, static_cast<cudaStream_t>(stream)));
}

int32_t tqd_op_wait_selftest(void* stream, uint32_t* err_bits_out) {
  if (!err_bits_out) return TQD_ERR_BAD_ARG;
  uint32_t bits = 0u;
  const cudaError_t e = run_wait_selftest(&bits, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return status_of(e);
  *err_bits_out = bits;
  return bits ? TQD_ERR_DEVICE_TIMEOUT : TQD_OK;
}

int32_t tqd_op_silu_mul(const float* g, const float* u, int64_t n, float* out, void* stream) {
  if (!g || !u || !out || n <= 0) return TQD_ERR_BAD_ARG;
  return status_of(launch_op_silu_mul(g, u, n, out, static_cast<cudaStream_t>(stream)));
}

size_t tqd_argmax_scratch_bytes(void) { return static_cast<size_t>(kOpArgmaxBlocks) * 8 + 16; }

int32_t tqd_op_argmax(const float* x, int64_t n, int32_t* idx_out, void* scratch, void* stream) {
  if (!x || !idx_out || !scratch || n <= 0 || n > 0x7FFFFFFEll) return TQD_ERR_BAD_ARG;
  float* cv = static_cast<float*>(scratch);
  int32_t* ci = reinterpret_cast<int32_t*>(cv + kOpArgmaxBlocks);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(ci + kOpArgmaxBlocks);
  return status_of(launch_op_argmax(x, n, idx_out, cv, ci, cnt, static_cast<cudaStream_t>(stream)));
}

size_t tqd_sample_scratch_bytes(int32_t vocab) {
  if (vocab <= 0) return 0;
  const size_t v4 = (static_cast<size_t>(vocab) + 3) / 4 * 4;
  return 384 + 3 * 4 * v4;
}

int32_t tqd_op_sample(const float* logits, int32_t vocab, int32_t* tokens, int32_t n_inputs,
                      const tqd_sampling* sampling, void* scratch, void* stream) {
  if (!logits || !tokens || !scratch || vocab <= 0 || n_inputs < 1 || n_inputs >= 0x7FFFFFFF ||
      reinterpret_cast<uintptr_t>(scratch) % 16)
    return TQD_ERR_BAD_ARG;
  SampleArgs a{};
  bool greedy = false;
  int32_t rc = sampling_args(sampling, a, &greedy);
  if (rc) return rc;
  if (greedy) a.temperature = 0.f;
  // scratch: the sequence descriptor and its state, then the padded logits,
  // the penalised logits and the input counts ([vocab rounded up to 4] each)
  const size_t v4 = (static_cast<size_t>(vocab) + 3) / 4 * 4;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  DevSeq* dseq = reinterpret_cast<DevSeq*>(base);
  DevState* dstate = reinterpret_cast<DevState*>(base + 256);
  float* lg = reinterpret_cast<float*>(base + 384);
  DevSeq h{};
  h.state = dstate;
  h.tokens = tokens;
  h.logits = lg;
  h.sz = lg + v4;
  h.scnt = reinterpret_cast<uint32_t*>(lg + 2 * v4);
  static_assert(sizeof(DevSeq) <= 256, "descriptor fits the scratch header");
  DevState st{static_cast<uint32_t>(n_inputs), 0u, 0u, 0u};
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // copies from pageable host memory are staged before cudaMemcpyAsync returns
  cudaError_t e = cudaMemcpyAsync(dseq, &h, sizeof(h), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(dstate, &st, sizeof(st), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(lg, logits, 4ull * vocab, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h.scnt, 0, 4 * v4, s);
  if (e == cudaSuccess) e = launch_sample(dseq, 1, vocab, n_inputs, a, s);
  return status_of(e);
}

}  // extern "C"
