/*
 * tqd.h — C ABI of libtqd, a GPU-resident greedy decoder for Qwen3-shaped
 * models with Q8_0 (or bf16) weights, built for sm_103a (GB300).
 *
 * What the library computes is the per-token decode step described by the
 * inferno.rs blog, "IV.4: One command buffer per token": embed the input
 * token, run every layer (RMSNorm, Q/K/V projections, per-head QK-norm, RoPE,
 * append to the KV cache, GQA attention, output projection + residual,
 * RMSNorm, gate/up projections, SwiGLU, down projection + residual), then the
 * final norm, the lm_head projection and the argmax, with weights and KV
 * cache resident on the GPU and only the next token id read back
 * (sections "Eight kernels" and "One command buffer").  The bf16 variant is
 * the Llama-style step without QK-norm of "Adding Metal to my Rust LLM engine",
 * section "What the kernels do".
 *
 * Conventions for every call:
 *  - Every function except tqd_destroy and tqd_status_name returns an
 *    int32_t status (TQD_OK = 0).  Arguments are validated before any GPU
 *    work; a refused call changes nothing.
 *  - Host pointers are owned by the caller and are never retained past the
 *    call.  All device memory is owned by the library (one arena per model,
 *    allocated by tqd_create, freed by tqd_destroy).  Functions named
 *    tqd_op_* take DEVICE pointers owned by the caller instead.
 *  - `stream` arguments are cudaStream_t values passed as void*.  A model
 *    runs all its work on the stream given to tqd_create; when that is NULL
 *    the model creates a private non-blocking stream and destroys it in
 *    tqd_destroy.  Operator entry points run on the stream given (NULL = the
 *    legacy default stream).
 *  - After TQD_ERR_CUDA or TQD_ERR_DEVICE_TIMEOUT a model is poisoned: every
 *    later call but tqd_destroy returns TQD_ERR_POISONED.
 *  - A model is not thread-safe: calls on one model must not overlap.
 */
#ifndef TQD_H
#define TQD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tqd_status {
  TQD_OK = 0,
  TQD_ERR_BAD_ARG = 1,             /* NULL pointer, out-of-range id, bad size */
  TQD_ERR_UNSUPPORTED_CONFIG = 2,  /* a config the library cannot run; see tqd_last_error() */
  TQD_ERR_NO_DEVICE = 3,           /* no CUDA device, or not an sm_103 device */
  TQD_ERR_CUDA = 4,                /* a CUDA runtime call failed (model poisoned) */
  TQD_ERR_OOM = 5,                 /* device allocation failed (nothing leaked) */
  TQD_ERR_CAPACITY = 6,            /* position would exceed max_seq */
  TQD_ERR_POS_MISMATCH = 7,        /* pos is not the sequence's next position */
  TQD_ERR_DEVICE_TIMEOUT = 8,      /* a bounded device-side wait gave up (model poisoned) */
  TQD_ERR_NUMERIC = 9,             /* every logit was NaN: no argmax exists */
  TQD_ERR_POISONED = 10,           /* an earlier fatal error; only tqd_destroy is valid */
  TQD_ERR_NOT_PREFILLED = 11       /* no step has produced logits for the sequence's next position */
} tqd_status;

enum { TQD_WEIGHT_Q8_0 = 0, TQD_WEIGHT_BF16 = 1 };

/* Execution schedule of one decode step (both compute the same thing):
 *  TQD_SCHED_GRAPH       one CUDA graph per token, one kernel per fused phase
 *  TQD_SCHED_PERSISTENT  one cooperative persistent kernel per token (or per
 *                        tqd_generate call), phases separated by bounded grid
 *                        barriers. */
enum { TQD_SCHED_GRAPH = 0, TQD_SCHED_PERSISTENT = 1 };

/* Element type of the KV cache.  TQD_KV_F32: the pages' f32 cache.
 * TQD_KV_F16: every K and V element rounded to the nearest IEEE binary16
 * (ties to even) when it is appended or uploaded, halving the attention's
 * bytes (the packed-F16 KV representation "Metal LLM decode" names as the
 * batched prefill+decode arm's next step).  Every entry point runs either
 * type: both batch-1 schedules, the batched step and the prefill tiles read
 * and append f16 rows when the cache is f16, the step's own row included
 * (rounded before it is used). */
enum { TQD_KV_F32 = 0, TQD_KV_F16 = 1 };

/* Model hyper-parameters ("One command buffer per token", section "The seam":
 * the plan's hidden, heads, kv heads, head_dim, intermediate, vocab, rms_eps,
 * rope_theta), plus this library's capacity fields. */
typedef struct tqd_config {
  int32_t n_layers;
  int32_t hidden;        /* H; Q8_0 needs H % 32 == 0, bf16 needs H % 8 == 0 */
  int32_t n_heads;       /* query heads */
  int32_t n_kv_heads;    /* key/value heads; n_heads % n_kv_heads == 0 */
  int32_t head_dim;      /* 64 or 128 */
  int32_t intermediate;  /* SwiGLU width I */
  int32_t vocab;         /* V; the lm_head has V rows */
  int32_t qk_norm;       /* 1: per-head RMSNorm of q and k before RoPE (Qwen3) */
  int32_t weight_type;   /* TQD_WEIGHT_Q8_0 or TQD_WEIGHT_BF16 */
  float rope_theta;
  float rms_eps;
  int32_t max_seq;       /* KV rows per sequence (positions 0 .. max_seq-1) */
  int32_t max_batch;     /* sequences held by the model (each its own KV) */
  int32_t schedule;      /* TQD_SCHED_* */
  int32_t kv_type;       /* TQD_KV_*; f16 needs a shape the batched step supports */
} tqd_config;

/* One layer's weights on the host.  Matrices are row-major [rows x cols]:
 *  Q8_0: rows * cols/32 blocks of 34 bytes (f16 scale little-endian, then 32
 *        int8 quants), row after row — the block of "Eight kernels";
 *  bf16: rows * cols uint16 bit patterns.
 * Shapes: wq [n_heads*head_dim x H], wk, wv [n_kv_heads*head_dim x H],
 * wo [H x n_heads*head_dim], w_gate, w_up [I x H], w_down [H x I].
 * Norm gains are f32: attn_norm, ffn_norm [H]; q_norm, k_norm [head_dim]
 * (ignored, may be NULL, when qk_norm == 0). */
typedef struct tqd_layer_weights {
  const float* attn_norm;
  const void* wq;
  const void* wk;
  const void* wv;
  const void* wo;
  const float* q_norm;
  const float* k_norm;
  const float* ffn_norm;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
} tqd_layer_weights;

typedef struct tqd_host_weights {
  const tqd_layer_weights* layers; /* [n_layers] */
  const float* out_norm;           /* [H] */
  const void* lm_head;             /* [V x H], same format as the layers */
  const void* embed;               /* [V x H] token embedding; NULL = tied to lm_head */
} tqd_host_weights;

typedef struct tqd_model tqd_model;

/* Create a model whose weights are the seeded synthetic ones the tests and
 * the benchmark use, in one call ("Metal LLM decode", section "Functions":
 * one call stands up the session): every matrix
 * N(0, 0.02), quantized to Q8_0 (scale = max|w| / 127 as f16, quants
 * rint(w / scale) clamped to +-127) or rounded to bf16, every norm gain
 * 1 + N(0, 0.1) in f32, the lm_head tied to the embedding.  Draws come from
 * counter-based splitmix64 streams, one per tensor: the lm_head 0, then per
 * layer attn_norm, wq, wk, wv, wo, q_norm, k_norm, ffn_norm, w_gate, w_up,
 * w_down, then the final norm; a normal draw is the Irwin-Hall sum of twelve
 * 16-bit uniforms.  The bytes equal those of the repository's Python
 * generator (synth.make_model(cfg, seed)).  Host memory for one copy of the
 * weights is held during the call.  Errors as tqd_create. */
int32_t tqd_create_synthetic(const tqd_config* cfg, uint64_t seed, void* stream, tqd_model** out);

/* Copy a model's weights back to host memory in the upload format of
 * tqd_host_weights (34-byte Q8_0 blocks or bf16, f32 gains): every pointer
 * of *out and of out->layers[0 .. n_layers) names caller memory of the
 * tensor's size (q_norm, k_norm only when qk_norm; embed may be NULL, and is
 * skipped when the model's embedding is tied).  Synchronous; off the decode
 * path.  Errors: BAD_ARG (a NULL destination), CUDA, POISONED. */
int32_t tqd_export_weights(tqd_model* model, const tqd_host_weights* out);

/* Name of a status code ("TQD_OK", ...); "TQD_UNKNOWN_STATUS" for others.
 * Needs no device.  ("Metal LLM decode", section "Status codes and the
 * dispatch budget": a status-name call that works on any host.) */
const char* tqd_status_name(int32_t status);

/* Human-readable detail of the last refusal on this thread (e.g. every
 * mismatched config field); "" when none.  Valid until the next call. */
const char* tqd_last_error(void);

/* Validate cfg, allocate the device arena (weights, KV cache for max_batch
 * sequences, activations, RoPE cos/sin table), upload and repack the weights
 * once, and prepare the per-token schedule.  On success *out owns the model.
 * Errors: BAD_ARG, UNSUPPORTED_CONFIG (nothing touched the GPU), NO_DEVICE,
 * OOM, CUDA.  ("One command buffer per token", GpuDecoder::try_new in
 * section "Resident state": upload once, allocate scratch once.) */
int32_t tqd_create(const tqd_config* cfg, const tqd_host_weights* weights, void* stream,
                   tqd_model** out);

/* Free everything the model owns.  NULL-safe.  Synchronises the model's stream. */
void tqd_destroy(tqd_model* model);

/* Forget sequence `seq`'s history: its next position becomes 0. */
int32_t tqd_reset(tqd_model* model, int32_t seq);

/* Drop positions n_pos .. next_pos-1 of sequence seq (0 <= n_pos <=
 * next_pos): the KV rows of positions below n_pos are kept, so decoding can
 * resume from a prefilled prompt without prefilling it again.
 * Errors: BAD_ARG. */
int32_t tqd_truncate(tqd_model* model, int32_t seq, int32_t n_pos);

/* The sequence's next position (number of filled KV rows). */
int32_t tqd_next_pos(tqd_model* model, int32_t seq, int32_t* pos_out);

/* Run the prompt ids[0..n-1] through the decoder on the GPU at positions
 * next_pos .. next_pos+n-1 (the decode step repeated, which is the same
 * computation as causal attention over the prompt), then write the greedy
 * next token to *next_out.  Errors: BAD_ARG (n <= 0, id out of range),
 * CAPACITY. */
int32_t tqd_prefill(tqd_model* model, int32_t seq, const int32_t* ids, int32_t n,
                    int32_t* next_out);

/* The same result as tqd_prefill (the prompt at next_pos .. next_pos+n-1,
 * then the greedy next token in *next_out), computed in tiles of up to 16
 * prompt positions: each tile is one batched step whose slots are the tile's
 * positions, so the projections sweep the weights once per tile on the tensor
 * cores (as tqd_decode_step_batch) and every slot attends to the cache rows
 * up to its own position, the tile's earlier rows included; the lm_head runs
 * for the prompt's last position only.  A longer prompt runs tile after tile,
 * each writing the next slice of the KV cache at its own offset ("Metal LLM
 * decode", the batched prefill+decode arm: prefill_batch, chunked calls at
 * position offsets).  Any max_batch; errors: as tqd_prefill, plus
 * UNSUPPORTED_CONFIG for a shape the batched kernels do not cover. */
int32_t tqd_prefill_batch(tqd_model* model, int32_t seq, const int32_t* ids, int32_t n,
                          int32_t* next_out);

/* Replace sequence seq's KV cache with n_pos host rows: k, v are f32
 * [n_layers][n_pos][n_kv_heads*head_dim] holding post-RoPE keys and values
 * ("One command buffer per token", section "The cache comes over once").
 * Sets next_pos = n_pos.  Errors: BAD_ARG, CAPACITY. */
int32_t tqd_kv_upload(tqd_model* model, int32_t seq, int32_t n_pos, const float* k,
                      const float* v);

/* One greedy decode step: feed `token` at position `pos`, which must equal
 * the sequence's next position, append its K/V row, and write the argmax of
 * the logits (ties to the lowest index, NaN never wins) to *next_out.  With
 * the persistent schedule the token travels as a launch argument and the next
 * token comes back inside the sequence's 16-byte state record (one launch and
 * one readback per call); the graph schedule copies the token up (4 bytes)
 * and reads the state back.  Errors: BAD_ARG, POS_MISMATCH, CAPACITY,
 * NUMERIC (all logits NaN).  ("One command buffer per token", section "One
 * command buffer": decode_step.) */
int32_t tqd_decode_step(tqd_model* model, int32_t seq, int32_t token, int32_t pos,
                        int32_t* next_out);

/* n_steps chained greedy steps: the first feeds first_token at next_pos, each
 * later one feeds the previous argmax, entirely on the device (no host
 * round trip between steps).  ids_out[i] receives the i-th generated id.
 * Errors: as tqd_decode_step. */
int32_t tqd_generate(tqd_model* model, int32_t seq, int32_t first_token, int32_t n_steps,
                     int32_t* ids_out);

/* One greedy step for sequences 0 .. n_seq-1 together (n_seq <= max_batch,
 * at most 64): sequence b feeds tokens[b] at pos[b] (its next position; the
 * positions may all differ).  The projections run as tensor-core contractions
 * over the batch (tcgen05, f32-accurate: exact int8 weight operands,
 * activations split into bf16 or f16 parts), attention per sequence.  Up to 16
 * sequences share one sweep of the weights; a larger batch runs as
 * consecutive groups of 16 (sequences 0-15, 16-31, ...), one sweep each.
 * next_out[b] receives sequence b's argmax.  Errors: as tqd_decode_step, plus
 * UNSUPPORTED_CONFIG when the model has no batched step (max_batch == 1).
 * ("Metal LLM decode", the batched prefill+decode arm: sequences share one
 * sweep of the weights per step, up to BATCH_DECODE_MAX_SEQS = 32.) */
int32_t tqd_decode_step_batch(tqd_model* model, int32_t n_seq, const int32_t* tokens,
                              const int32_t* pos, int32_t* next_out);

/* n_steps chained batched greedy steps for sequences 0 .. n_seq-1, each
 * starting from first_tokens[b] at its next position; ids_out[i * n_seq + b]
 * receives step i's id of sequence b. */
int32_t tqd_generate_batch(tqd_model* model, int32_t n_seq, const int32_t* first_tokens,
                           int32_t n_steps, int32_t* ids_out);

/* Controls of seeded sampling ("Metal LLM decode", the sampled arm of the
 * batched prefill+decode section, which names them and fixes that
 * temperature <= 0 falls back to the greedy token and top_k = 1 reproduces
 * it).  The draw, in this order: the penalties on the distinct tokens among
 * the sequence's inputs so far (count c): l = l > 0 ? l / repeat : l * repeat,
 * then l -= presence, then l -= frequency * c (NaN logits count as -inf);
 * the tokens are ranked by that penalised l, descending, ties to the lower
 * index (division by a positive temperature keeps the order, so ranking
 * before it keeps top_k = 1 the greedy token even where l / temperature
 * merges two logits); top_k keeps the first top_k of that order; top_p keeps,
 * of those, the shortest prefix of the order whose probability reaches top_p
 * of their total; min_p keeps z - z_max >= ln(min_p), z = l / temperature;
 * the token is drawn from the kept probabilities exp(z - z_max) by inverting
 * their running sum in index order at u = the top 24 bits of splitmix64's
 * output number `position` from `seed`, times 2^-24, where position is the
 * drawn token's position.  Every float step is f32; the probabilities are
 * summed as integers in units of 2^-32 of the most likely token's, so a draw
 * is deterministic.  A temperature so small that l_max / temperature
 * overflows f32 draws the greedy token of the penalised logits (the limit
 * of the distribution as the temperature goes to 0). */
typedef struct tqd_sampling {
  float temperature;        /* <= 0: the greedy token */
  int32_t top_k;            /* 0: off; 1: the greedy token of the penalised logits */
  float top_p;              /* (0, 1]; 1: off */
  float min_p;              /* [0, 1]; 0: off */
  float repeat_penalty;     /* > 0; 1: off */
  float presence_penalty;   /* 0: off */
  float frequency_penalty;  /* 0: off */
  uint64_t seed;
} tqd_sampling;

/* Draw the token for sequence seq's next position from its last step's
 * logits (after a prefill or a decode step) and make it the sequence's input
 * there; *token_out receives it.  Errors: BAD_ARG (controls out of range,
 * non-finite), NOT_PREFILLED (no logits for the next position: nothing run
 * since create, reset, truncate or kv_upload). */
int32_t tqd_sample(tqd_model* model, int32_t seq, const tqd_sampling* sampling, int32_t* token_out);

/* As tqd_generate, with every step's token drawn under `sampling` instead of
 * the argmax, on the device (the draw runs after each step; no host round
 * trip between steps).  With 1 <= top_k <= 64 the draw takes two passes: one
 * block per 1024-token vocabulary slice keeps the slice's first top_k, one
 * block merges them; otherwise one block per sequence draws from the whole
 * vocabulary.  Both give the same token. */
int32_t tqd_generate_sampled(tqd_model* model, int32_t seq, int32_t first_token, int32_t n_steps,
                             const tqd_sampling* sampling, int32_t* ids_out);

/* As tqd_generate_batch, with every sequence's token drawn under `sampling`
 * (the draw of every sequence after each batched step, as in
 * tqd_generate_sampled). */
int32_t tqd_generate_batch_sampled(tqd_model* model, int32_t n_seq, const int32_t* first_tokens,
                                   int32_t n_steps, const tqd_sampling* sampling, int32_t* ids_out);

/* Copy the logits of sequence seq's last step (f32 [vocab]) to host_out.
 * A debugging and parity hook, off the decode path ("One command buffer per
 * token", read_logits). */
int32_t tqd_read_logits(tqd_model* model, int32_t seq, float* host_out);

/* Number of device phases one decode step runs (kernel launches for
 * TQD_SCHED_GRAPH: 5 per layer plus 2; for TQD_SCHED_PERSISTENT the dependent
 * phases of one step: per layer the projections, the attention chunks, the O
 * projection and the fused feed-forward, then the lm_head: 4 per layer plus
 * 1) — the analogue of the per-token dispatch budget of "Metal LLM decode". */
int32_t tqd_phase_count(tqd_model* model, int32_t* out);

/* Algorithmic HBM bytes of one decode step at position pos (weights read
 * once, pos+1 KV rows read per layer, one KV row written per layer). */
int32_t tqd_step_bytes(tqd_model* model, int32_t pos, int64_t* bytes_out);

/* ------------------------------------------------------------------------
 * Operator entry points (device pointers, caller-owned, on `stream`).
 * They run the same device code as the decode step, one phase at a time, so
 * each can be checked on its own ("The correctness ladder", rung one).
 * All return BAD_ARG for NULL pointers or unsupported sizes, CUDA on a launch
 * failure; they allocate nothing.
 * ------------------------------------------------------------------------ */

/* Repack a Q8_0 matrix from 34-byte blocks (rows x cols/32 blocks) into the
 * library's row layout: per row, cols int8 quants then cols/32 f16 scales,
 * padded to a multiple of 16 bytes (cols * 17/16 bytes when cols % 256 == 0;
 * cols % 32 == 0). */
int32_t tqd_op_q8_0_repack(const uint8_t* w_blocks, int64_t rows, int64_t cols, uint8_t* w_rows,
                           void* stream);

/* y[r] = sum_b scale_rb * sum_j quant_rbj * x[32b+j] over a repacked Q8_0
 * matrix ("Eight kernels", q8_matvec).  x f32 [cols], y f32 [rows]. */
int32_t tqd_op_q8_0_matvec(const uint8_t* w_rows, int64_t rows, int64_t cols, const float* x,
                           float* y, void* stream);

/* y = W x for a bf16 matrix [rows x cols] (cols % 8 == 0). */
int32_t tqd_op_bf16_matvec(const uint16_t* w, int64_t rows, int64_t cols, const float* x,
                           float* y, void* stream);

/* out[r] = x[r] * (mean(x[r]^2) + eps)^(-1/2) * g for `rows` rows of n
 * ("Eight kernels", rms_norm_row).  n <= 16384. */
int32_t tqd_op_rmsnorm(const float* x, const float* g, int32_t rows, int32_t n, float eps,
                       float* out, void* stream);

/* Fill table [max_pos][head_dim/2] of (cos a, sin a) f32 pairs with
 * a = p * theta^(-i/(head_dim/2)), computed in f64 on the device. */
int32_t tqd_op_rope_table(float theta, int32_t head_dim, int32_t max_pos, float* table,
                          void* stream);

/* Half-split RoPE in place on n_heads heads of x at position pos, using a
 * table from tqd_op_rope_table ("Eight kernels", rope_row). */
int32_t tqd_op_rope(float* x, int32_t n_heads, int32_t head_dim, int32_t pos, const float* table,
                    void* stream);

/* Split-K decode attention ("Eight kernels", attention_decode, restated as a
 * flash-decode over n_chunks key ranges with a log-sum-exp combine):
 * q f32 [n_heads*hd], K, V f32 [S][n_kv*hd], out f32 [n_heads*hd].
 * `scratch` is caller-owned device memory of
 * tqd_attention_scratch_bytes(n_heads, n_kv, hd, n_chunks) bytes; the call
 * leaves it ready for reuse.  hd must be 64 or 128; 1 <= n_chunks <= 1024. */
int32_t tqd_op_attention(const float* q, const float* K, const float* V, int32_t S,
                         int32_t n_heads, int32_t n_kv, int32_t head_dim, int32_t n_chunks,
                         float* out, void* scratch, void* stream);
size_t tqd_attention_scratch_bytes(int32_t n_heads, int32_t n_kv, int32_t head_dim,
                                   int32_t n_chunks);

/* Failure detection without a GPU fault: runs one block whose bounded device
 * waits cannot complete (an mbarrier no thread arrives at, and a counter that
 * nothing increments, polled the way a grid barrier is); each gives up after
 * its 2 s limit, records its error bit and returns.  *err_bits_out receives
 * the bits (1: counter wait, 2: mbarrier wait); the status is
 * TQD_ERR_DEVICE_TIMEOUT when any is set.  The CUDA context stays usable.
 * Takes about 2 s ("One command buffer per token", "The seam": a failed step
 * is reported, not hung on). */
int32_t tqd_op_wait_selftest(void* stream, uint32_t* err_bits_out);

/* out = silu(g) * u elementwise, silu(z) = z / (1 + e^-z)
 * ("Eight kernels", silu_hadamard). */
int32_t tqd_op_silu_mul(const float* g, const float* u, int64_t n, float* out, void* stream);

/* *idx_out = index of the largest x (ties -> lowest index, NaN never wins,
 * -1 when all NaN) ("Eight kernels", argmax_row).  scratch: caller-owned
 * device memory of tqd_argmax_scratch_bytes() bytes. */
int32_t tqd_op_argmax(const float* x, int64_t n, int32_t* idx_out, void* scratch, void* stream);
size_t tqd_argmax_scratch_bytes(void);

/* Seeded sampling on caller memory, the draw of tqd_sample (controls and
 * order as documented at tqd_sampling): logits f32 [vocab] (device); tokens
 * int32 [n_inputs + 1] (device): tokens[0, n_inputs) are the inputs so far
 * (the penalties' history) and the drawn token, for position n_inputs, is
 * written to tokens[n_inputs] (-1 when every logit is NaN).  n_inputs >= 1.
 * scratch: caller-owned device memory of tqd_sample_scratch_bytes(vocab)
 * bytes (the logits are copied there, padded for 16-byte loads).  BAD_ARG
 * for out-of-range controls as tqd_sample. */
int32_t tqd_op_sample(const float* logits, int32_t vocab, int32_t* tokens, int32_t n_inputs,
                      const tqd_sampling* sampling, void* scratch, void* stream);
size_t tqd_sample_scratch_bytes(int32_t vocab);

/* Allocation-free variant of tqd_op_attention (the pages have no counterpart;
 * this is an interface for callers that may not allocate device memory while
 * they run, e.g. a serving loop whose memory budget is fixed at start-up, or a
 * host thread that must not trigger the device-wide synchronisation that
 * cudaMalloc / cudaFree can cause).  Same inputs, output and result as
 * tqd_op_attention; the per-chunk scratch lives in a static device array of
 * tqd_op_attention_noalloc_max_scratch() bytes (1 MiB) that every device
 * loading the library holds until the process exits.  No device memory is
 * allocated by the call.
 *  - The first call on a device looks up that array's device address (with
 *    the device current); make that first call before any stream capture.
 *    A lookup that fails returns TQD_ERR_CUDA and is tried again by the
 *    next call; only a successful one is kept.
 *  - Calls whose tqd_attention_scratch_bytes(...) exceeds the array's size
 *    return TQD_ERR_BAD_ARG (see tqd_last_error()).
 *  - Every call on a device shares the array and leaves its contents behind;
 *    the call clears the arrival counters it needs on `stream` before its
 *    kernel.  Calls that overlap on the GPU (other streams, or concurrent
 *    host threads) race on the array and must be serialised by the caller. */
int32_t tqd_op_attention_noalloc(const float* q, const float* K, const float* V, int32_t S,
                                 int32_t n_heads, int32_t n_kv, int32_t head_dim,
                                 int32_t n_chunks, float* out, void* stream);
size_t tqd_op_attention_noalloc_max_scratch(void);

#ifdef __cplusplus
}
#endif

#endif /* TQD_H */
