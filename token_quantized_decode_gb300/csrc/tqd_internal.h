// Host-side interface between the engine / operator entry points and the
// kernels translation unit.  Every launcher returns the cudaError_t of the
// launch; none synchronises.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "tqd_device.cuh"

struct tqd_sampling;  // include/tqd.h

namespace tqd {

constexpr int kMatvecThreads = 256;      // 8 warps per matvec block (graph schedule)
constexpr int kAttnThreads = 128;        // 4 warps per attention block (graph schedule)
constexpr int kMaxArgmaxBlocks = 2048;   // bound on lm_head blocks (argmax candidates)

// Chunks of 16 bytes per lane needed for a row of K weights, rounded up to an
// instantiated value; 0 when K is too long for the matvec kernels.
__host__ __device__ inline int matvec_cpl(int fmt, int K) {
  const int epc = fmt == 0 ? 16 : 8;
  if (K <= 0 || K % epc) return 0;
  const int need = (K / epc + 31) / 32;
  if (need <= 2) return need;
  if (need <= 4) return 4;
  if (need <= 6) return 6;
  if (need <= 8) return 8;
  if (need <= 12) return 12;
  return 0;
}

// Bytes of one stored Q8_0 row of K weights: K quants, K/32 f16 scales,
// padded to a multiple of 16 bytes (no padding when K % 256 == 0).
__host__ __device__ inline size_t q8_row_bytes(int64_t K) {
  return static_cast<size_t>((K + K / 16 + 15) / 16 * 16);
}

// Shared memory (bytes) of the matvec kernel for K columns.
__host__ __device__ inline size_t matvec_smem_bytes(int K) {
  const int kpad = (K + 3) & ~3;
  return static_cast<size_t>(kpad) * 4 + 64 * 4 + 16;
}

struct MatvecLaunch {
  const uint8_t* W;
  size_t row_bytes;
  int K, rows, epi;
  float* y;
  const float* src;     // vector staged into shared memory (K floats)
  const float* norm_g;  // RMSNorm gain applied to the staged vector, or nullptr
  float eps;
  // lm_head only: the step's argmax epilogue
  bool lm_head;
  DevSeq seq;
  int max_seq;
};

cudaError_t launch_matvec(int fmt, const MatvecLaunch& a, int blocks, cudaStream_t st, bool pdl);

cudaError_t launch_embed(const DevModel& m, const DevSeq& s, cudaStream_t st, bool pdl);
cudaError_t launch_attention(const DevModel& m, const DevSeq& s, int layer, cudaStream_t st,
                             bool pdl);
cudaError_t launch_advance(const DevSeq& s, cudaStream_t st, bool pdl);

// One cooperative launch running n_steps decode steps (the last `full_steps`
// of them with the lm_head and argmax; earlier ones are prefill positions).
cudaError_t launch_persistent(const DevModel& m, const DevSeq& s, int n_steps, int full_from,
                              int blocks, cudaStream_t st);
int persistent_blocks_per_sm(const DevModel& m);  // 0: unsupported or not resident
bool persistent_supported(const DevModel& m);
size_t persistent_smem_bytes(const DevModel& m);

// Set-up kernels.
cudaError_t launch_q8_repack(const uint8_t* src_blocks, int64_t rows, int64_t cols, uint8_t* dst,
                             int64_t dst_row0, int64_t dst_row_step, cudaStream_t st);
cudaError_t launch_rope_table(double theta, int head_dim, int max_pos, float2* table,
                              cudaStream_t st);

// Operator entry points' kernels.
cudaError_t launch_op_matvec(int fmt, const uint8_t* W, size_t row_bytes, int rows, int K,
                             const float* x, float* y, cudaStream_t st);
cudaError_t launch_op_rmsnorm(const float* x, const float* g, int rows, int n, float eps,
                              float* out, cudaStream_t st);
cudaError_t launch_op_rope(float* x, int n_heads, int head_dim, const float2* row,
                           cudaStream_t st);
cudaError_t launch_op_attention(const float* q, const float* K, const float* V, int S, int nq,
                                int nkv, int hd, int n_chunks, float* out, float* part_o,
                                float* part_ml, uint32_t* count, cudaStream_t st);
cudaError_t launch_op_silu_mul(const float* g, const float* u, int64_t n, float* out,
                               cudaStream_t st);
cudaError_t launch_op_argmax(const float* x, int64_t n, int32_t* out, float* cand_v,
                             int32_t* cand_i, uint32_t* count, cudaStream_t st);
constexpr int kOpArgmaxBlocks = 304;

bool attention_supported(int hd, int group);

// Batched step (tqd_batch.cu): up to batch_max() sequences per step, tcgen05
// contractions for the projections, streaming split-K attention.
int batch_max();
int batch_ss_slots(int H);  // partial sums of squares per activation ([slots][batch_max()])
bool batch_supported(const DevModel& m);
cudaError_t batch_setup(const DevModel& m);
// The lm_head in the tile-pass order the batched step streams: its size, and
// the kernel that writes it from the row layout.
size_t batch_head_bytes(int rows, int K, int fmt);
cudaError_t launch_head_tile(const uint8_t* rows_src, size_t rb, int rows, int K, int fmt, uint8_t* dst,
                             cudaStream_t st);
// One upload of a step's host tokens for all sequences (tok[b] -> sequence b's
// input at its next position), and one readback of every sequence's argmax and
// error word after the step (out[b], out[n + b]).
cudaError_t launch_batch_tokens_in(const DevSeq* seqs, int n, const int32_t* tok, cudaStream_t st);
cudaError_t launch_batch_tokens_out(const DevSeq* seqs, int n, int32_t* out, cudaStream_t st);
// A prefill tile's slot positions (slot b at the sequence's next position + b)
// before the tile, and after it the sequence's advance by n and the slots'
// error bits.  slots: batch_max() + 1 descriptors, the last the sequence's own.
cudaError_t launch_prefill_tile_begin(const DevSeq* slots, int n, cudaStream_t st);
cudaError_t launch_prefill_tile_end(const DevSeq* slots, int n, cudaStream_t st);
// PO / PML: the attention's chunk partials, [n][nq][nch][hd] and [n][nq][nch][2].
// tile: seqs are the slots of one sequence's prefill tile (K/V rows appended
// before the attention); out0: the first slot whose logits and argmax are
// produced (0 for a decode step; >= n skips the lm_head).
cudaError_t enqueue_batch_step(const DevModel& m, const DevLayer* host_layers, const uint8_t* lm_tiled,
                               const DevSeq* seqs, int n, int nch, float* X, float* QKV, float* PO, float* PML,
                               float* H, float* SS, uint32_t* count, uint32_t* err, cudaStream_t st, bool tile,
                               int out0);

// Seeded sampling (tqd_sample.cu): one block per sequence draws the token for
// its next position from its last logits and writes it there as the input.
struct SampleArgs {
  float temperature;   // <= 0: the greedy token of the raw logits
  int top_k;           // 1 <= top_k < V, else off
  float top_p;         // < 1, else off
  float ln_min_p;      // f32(ln(min_p)), -inf when off
  float repeat, presence, frequency;
  int penalize;        // any penalty differs from neutral
  unsigned long long seed;
  int parts;           // set by launch_sample: vocabulary slices whose top_k lists k_sample merges (0: none)
};
// Vocabulary entries per slice of the sampler's first pass, and the largest
// top_k that pass serves (per sequence: DevSeq::sparts holds
// ceil(V / kSampleSlice) * kSamplePartK keys).
constexpr int kSampleSlice = 1024;
constexpr int kSamplePartK = 64;
// Groups of batch_max() sequences a batched step can run (tqd_config.max_batch <= 64).
constexpr int kBatchGroups = 4;
// slices: the sequences' DevSeq::sparts hold the per-slice lists (the
// engine's sequences), so top_k <= kSamplePartK draws take the two-pass path.
cudaError_t launch_sample(const DevSeq* seqs, int n, int V, int max_seq, const SampleArgs& a, cudaStream_t st,
                          bool slices = false);
// Validate the caller's sampling controls into a, and say whether they are greedy.
int32_t sampling_args(const ::tqd_sampling* p, SampleArgs& a, bool* greedy);

// The bounded-wait self-test (tqd_op_wait_selftest): runs it on st and
// returns the error bits its waits set.
cudaError_t run_wait_selftest(uint32_t* err_bits, cudaStream_t st);

// Record the text tqd_last_error() returns on this thread.
void set_last_error(const char* msg);

}  // namespace tqd
