// Host engine and C ABI of libtqd (declarations and contracts in tqd.h).
//
// A model owns one device arena: repacked weights, the RoPE cos/sin table,
// and per sequence its KV cache, token history, activations and the
// split-K / argmax partials.  Weights are uploaded once; a decode step
// moves four bytes of token id each way ("One command buffer per token",
// sections "Resident state" and "One command buffer").
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "tqd.h"
#include "tqd_internal.h"

using namespace tqd;

namespace {

thread_local std::string g_last_error;

}  // namespace

void tqd::set_last_error(const char* msg) { g_last_error = msg; }

namespace {

void set_error(const char* fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct SeqSlot {
  DevSeq d{};
  int32_t next_pos = 0;
  int32_t logits_pos = -1;  // next_pos when the logits buffer was last written (they predict it)
  cudaGraphExec_t g_full = nullptr;
  cudaGraphExec_t g_layers = nullptr;
};

}  // namespace

struct tqd_model {
  tqd_config cfg{};
  cudaStream_t stream = nullptr;
  bool own_stream = false;  // created by tqd_create (caller passed NULL)
  int device = 0, num_sms = 0;
  uint8_t* arena = nullptr;
  size_t arena_bytes = 0;
  DevModel dm{};
  std::vector<SeqSlot> seqs;
  std::vector<DevLayer> host_layers;  // host copy of dm.layers (launch arguments)
  int32_t* h_tokens = nullptr;  // pinned staging [max(max_seq + 1, 256)]
  DevState* h_state = nullptr;  // pinned
  bool poisoned = false;
  bool pdl = true;
  int blocks_qkv = 0, blocks_o = 0, blocks_gu = 0, blocks_d = 0, blocks_lm = 0;
  int blocks_persist = 0;
  int64_t weight_bytes = 0;
  // batched step: activations of up to batch_max() sequences, the device copy
  // of the sequences' descriptors, one graph per batch size
  bool batch_ok = false;
  float *bx = nullptr, *bqkv = nullptr, *bpo = nullptr, *bpml = nullptr, *bh = nullptr;
  DevSeq* dseqs = nullptr;
  uint32_t* bcount = nullptr;
  float* bss = nullptr;
  uint8_t* blm = nullptr;  // the lm_head in the batched step's tile-pass order
  int32_t* bio = nullptr;  // a batched step's tokens in [16], argmax out and error words [2 x 16]
  // batches beyond batch_max() sequences run as consecutive groups of at most
  // batch_max(): one graph per (group, group size)
  cudaGraphExec_t bgraph[kBatchGroups][17] = {};
  // prefill tiles: batch_max() slot descriptors and the sequence's own (the
  // device copy and its host image), the slots' state words, and one graph per
  // (tile size, whether the tile ends the prompt)
  DevSeq* pslots = nullptr;
  std::vector<DevSeq> pslots_host;
  DevState* pstates = nullptr;
  cudaGraphExec_t pgraph[17][2] = {};
};

namespace {

int32_t fail_cuda(tqd_model* m, cudaError_t e, const char* what) {
  set_error("%s: %s", what, cudaGetErrorString(e));
  if (m) m->poisoned = true;
  return TQD_ERR_CUDA;
}

#define CK(call, what)                                  \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return fail_cuda(m, e_, what); \
  } while (0)

// Bytes of one stored row of a matrix with `cols` columns.
size_t row_bytes(int wtype, int cols) {
  return wtype == TQD_WEIGHT_Q8_0 ? q8_row_bytes(cols) : static_cast<size_t>(cols) * 2;
}
// Bytes of one host row (34-byte blocks for Q8_0).
size_t host_row_bytes(int wtype, int cols) {
  return wtype == TQD_WEIGHT_Q8_0 ? static_cast<size_t>(cols) / 32 * 34
                                  : static_cast<size_t>(cols) * 2;
}

int32_t validate_config(const tqd_config* c) {
  std::string bad;
  auto need = [&](bool ok, const char* msg) {
    if (!ok) {
      if (!bad.empty()) bad += "; ";
      bad += msg;
    }
  };
  need(c->n_layers >= 1, "n_layers must be >= 1");
  need(c->hidden >= 1, "hidden must be >= 1");
  need(c->n_heads >= 1 && c->n_kv_heads >= 1 && c->n_heads % c->n_kv_heads == 0,
       "n_heads must be a positive multiple of n_kv_heads");
  need(c->head_dim == 64 || c->head_dim == 128, "head_dim must be 64 or 128");
  if (c->n_kv_heads >= 1)
    need(attention_supported(c->head_dim == 64 ? 64 : 128, c->n_heads / c->n_kv_heads),
         "n_heads / n_kv_heads must be 1, 2, 3, 4 or 8");
  need(c->intermediate >= 1, "intermediate must be >= 1");
  need(c->vocab >= 1, "vocab must be >= 1");
  need(c->qk_norm == 0 || c->qk_norm == 1, "qk_norm must be 0 or 1");
  need(c->weight_type == TQD_WEIGHT_Q8_0 || c->weight_type == TQD_WEIGHT_BF16,
       "weight_type must be TQD_WEIGHT_Q8_0 or TQD_WEIGHT_BF16");
  need(c->max_seq >= 1 && c->max_seq <= (1 << 24), "max_seq must be in [1, 2^24]");
  need(c->max_batch >= 1 && c->max_batch <= 64, "max_batch must be in [1, 64]");
  need(c->kv_type == TQD_KV_F32 || c->kv_type == TQD_KV_F16, "kv_type must be TQD_KV_F32 or TQD_KV_F16");
  need(c->schedule == TQD_SCHED_GRAPH || c->schedule == TQD_SCHED_PERSISTENT,
       "schedule must be TQD_SCHED_GRAPH or TQD_SCHED_PERSISTENT");
  need(std::isfinite(c->rope_theta) && c->rope_theta > 0.f, "rope_theta must be > 0");
  need(std::isfinite(c->rms_eps) && c->rms_eps >= 0.f, "rms_eps must be >= 0");
  const int qw = c->n_heads * c->head_dim;
  if (c->weight_type == TQD_WEIGHT_Q8_0) {
    need(c->hidden % 32 == 0, "Q8_0 needs hidden % 32 == 0");
    need(qw % 32 == 0, "Q8_0 needs n_heads*head_dim % 32 == 0");
    need(c->intermediate % 32 == 0, "Q8_0 needs intermediate % 32 == 0");
  } else {
    need(c->hidden % 8 == 0, "bf16 needs hidden % 8 == 0");
    need(qw % 8 == 0, "bf16 needs n_heads*head_dim % 8 == 0");
    need(c->intermediate % 8 == 0, "bf16 needs intermediate % 8 == 0");
  }
  const int fmt = c->weight_type == TQD_WEIGHT_Q8_0 ? kFmtQ8 : kFmtBF16;
  if (bad.empty()) {
    need(matvec_cpl(fmt, c->hidden) != 0, "hidden too large for the matvec kernels");
    need(matvec_cpl(fmt, qw) != 0, "n_heads*head_dim too large for the matvec kernels");
    need(matvec_cpl(fmt, c->intermediate) != 0, "intermediate too large for the matvec kernels");
  }
  if (!bad.empty()) {
    set_error("unsupported config: %s", bad.c_str());
    return TQD_ERR_UNSUPPORTED_CONFIG;
  }
  return TQD_OK;
}

int32_t check_weights(const tqd_config* c, const tqd_host_weights* w) {
  if (!w->layers || !w->out_norm || !w->lm_head) {
    set_error("weights: layers, out_norm and lm_head are required");
    return TQD_ERR_BAD_ARG;
  }
  for (int l = 0; l < c->n_layers; ++l) {
    const tqd_layer_weights& L = w->layers[l];
    if (!L.attn_norm || !L.wq || !L.wk || !L.wv || !L.wo || !L.ffn_norm || !L.w_gate || !L.w_up ||
        !L.w_down || (c->qk_norm && (!L.q_norm || !L.k_norm))) {
      set_error("weights: layer %d has a NULL tensor", l);
      return TQD_ERR_BAD_ARG;
    }
  }
  return TQD_OK;
}

// Matvec blocks for `rows` rows with K columns on the graph schedule.
int matvec_blocks(int fmt, int rows, int K, int num_sms, int cap) {
  const int cpl = matvec_cpl(fmt, K);
  const int R = cpl >= 4 ? 2 : 8 / cpl;
  const int groups = (rows + R - 1) / R;
  int b = (groups + kMatvecThreads / 32 - 1) / (kMatvecThreads / 32);
  const int lim = cap > 0 ? cap : 4 * num_sms;
  if (b > lim) b = lim;
  return b < 1 ? 1 : b;
}

cudaError_t enqueue_step(tqd_model* m, SeqSlot& s, bool full) {
  const DevModel& dm = m->dm;
  const int fmt = dm.wtype;
  const bool pdl = m->pdl;
  cudaStream_t st = m->stream;
  cudaError_t e = launch_embed(dm, s.d, st, false);
  if (e != cudaSuccess) return e;
  const std::vector<DevLayer>& layers = m->host_layers;
  for (int l = 0; l < dm.n_layers; ++l) {
    const DevLayer& L = layers[l];
    MatvecLaunch a{};
    a.eps = dm.eps;
    a.seq = s.d;
    a.max_seq = dm.max_seq;
    // norm + QKV
    a.W = L.wqkv; a.row_bytes = dm.row_bytes_h; a.K = dm.H; a.rows = dm.qw + 2 * dm.kvw;
    a.epi = kEpiStore; a.y = s.d.qkv; a.src = s.d.x; a.norm_g = L.attn_norm; a.lm_head = false;
    if ((e = launch_matvec(fmt, a, m->blocks_qkv, st, pdl)) != cudaSuccess) return e;
    if ((e = launch_attention(dm, s.d, l, st, pdl)) != cudaSuccess) return e;
    // O + residual
    a.W = L.wo; a.row_bytes = dm.row_bytes_qw; a.K = dm.qw; a.rows = dm.H;
    a.epi = kEpiResid; a.y = s.d.x; a.src = s.d.attn; a.norm_g = nullptr;
    if ((e = launch_matvec(fmt, a, m->blocks_o, st, pdl)) != cudaSuccess) return e;
    // norm + gate/up + SwiGLU
    a.W = L.wgu; a.row_bytes = dm.row_bytes_h; a.K = dm.H; a.rows = 2 * dm.I;
    a.epi = kEpiSwiGLU; a.y = s.d.h; a.src = s.d.x; a.norm_g = L.ffn_norm;
    if ((e = launch_matvec(fmt, a, m->blocks_gu, st, pdl)) != cudaSuccess) return e;
    // down + residual
    a.W = L.wd; a.row_bytes = dm.row_bytes_i; a.K = dm.I; a.rows = dm.H;
    a.epi = kEpiResid; a.y = s.d.x; a.src = s.d.h; a.norm_g = nullptr;
    if ((e = launch_matvec(fmt, a, m->blocks_d, st, pdl)) != cudaSuccess) return e;
  }
  if (full) {
    MatvecLaunch a{};
    a.eps = dm.eps;
    a.seq = s.d;
    a.max_seq = dm.max_seq;
    a.W = dm.lm_head; a.row_bytes = dm.row_bytes_h; a.K = dm.H; a.rows = dm.V;
    a.epi = kEpiArgmax; a.y = s.d.logits; a.src = s.d.x; a.norm_g = dm.out_norm; a.lm_head = true;
    return launch_matvec(fmt, a, m->blocks_lm, st, pdl);
  }
  return launch_advance(s.d, st, pdl);
}

int32_t capture(tqd_model* m, SeqSlot& s, bool full, cudaGraphExec_t* out) {
  cudaGraph_t g = nullptr;
  CK(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal), "begin capture");
  cudaError_t e = enqueue_step(m, s, full);
  cudaError_t e2 = cudaStreamEndCapture(m->stream, &g);
  if (e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return fail_cuda(m, e, "capture step");
  }
  if (e2 != cudaSuccess) return fail_cuda(m, e2, "end capture");
  e = cudaGraphInstantiate(out, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) return fail_cuda(m, e, "instantiate graph");
  return TQD_OK;
}

// Enqueue n steps for sequence s; steps with index >= full_from run the
// lm_head and argmax.
int32_t run_steps(tqd_model* m, SeqSlot& s, int n, int full_from) {
  if (m->cfg.schedule == TQD_SCHED_PERSISTENT) {
    CK(launch_persistent(m->dm, s.d, n, full_from, m->blocks_persist, m->stream),
       "persistent launch");
    return TQD_OK;
  }
  if (!s.g_full) {
    int32_t rc = capture(m, s, true, &s.g_full);
    if (rc) return rc;
  }
  if (full_from > 0 && !s.g_layers) {
    int32_t rc = capture(m, s, false, &s.g_layers);
    if (rc) return rc;
  }
  for (int i = 0; i < n; ++i)
    CK(cudaGraphLaunch(i >= full_from ? s.g_full : s.g_layers, m->stream), "graph launch");
  return TQD_OK;
}

// Read the device state back, synchronise, and turn error bits into a status.
int32_t finish(tqd_model* m, SeqSlot& s) {
  CK(cudaMemcpyAsync(m->h_state, s.d.state, sizeof(DevState), cudaMemcpyDeviceToHost, m->stream),
     "read state");
  CK(cudaStreamSynchronize(m->stream), "synchronize");
  const uint32_t err = m->h_state->err;
  if (err == 0) return TQD_OK;
  if (err & (kErrGridBarrier | kErrMbarrier)) {
    m->poisoned = true;
    set_error("device wait timed out (error bits 0x%x)", err);
    return TQD_ERR_DEVICE_TIMEOUT;
  }
  // clear recoverable bits so the sequence can continue after a reset
  CK(cudaMemsetAsync(&s.d.state->err, 0, sizeof(uint32_t), m->stream), "clear error");
  CK(cudaStreamSynchronize(m->stream), "synchronize");
  if (err & kErrAllNaN) {
    set_error("every logit was NaN");
    return TQD_ERR_NUMERIC;
  }
  if (err & kErrCapacity) {
    set_error("position beyond max_seq");
    return TQD_ERR_CAPACITY;
  }
  set_error("token id outside the vocabulary");
  return TQD_ERR_BAD_ARG;
}

int32_t check_model(tqd_model* m, int32_t seq) {
  if (!m) {
    set_error("model is NULL");
    return TQD_ERR_BAD_ARG;
  }
  if (m->poisoned) {
    set_error("model is poisoned by an earlier fatal error");
    return TQD_ERR_POISONED;
  }
  if (seq < 0 || seq >= m->cfg.max_batch) {
    set_error("seq %d outside [0, %d)", seq, m->cfg.max_batch);
    return TQD_ERR_BAD_ARG;
  }
  return TQD_OK;
}

}  // namespace

extern "C" {

const char* tqd_status_name(int32_t s) {
  switch (s) {
    case TQD_OK: return "TQD_OK";
    case TQD_ERR_BAD_ARG: return "TQD_ERR_BAD_ARG";
    case TQD_ERR_UNSUPPORTED_CONFIG: return "TQD_ERR_UNSUPPORTED_CONFIG";
    case TQD_ERR_NO_DEVICE: return "TQD_ERR_NO_DEVICE";
    case TQD_ERR_CUDA: return "TQD_ERR_CUDA";
    case TQD_ERR_OOM: return "TQD_ERR_OOM";
    case TQD_ERR_CAPACITY: return "TQD_ERR_CAPACITY";
    case TQD_ERR_POS_MISMATCH: return "TQD_ERR_POS_MISMATCH";
    case TQD_ERR_DEVICE_TIMEOUT: return "TQD_ERR_DEVICE_TIMEOUT";
    case TQD_ERR_NUMERIC: return "TQD_ERR_NUMERIC";
    case TQD_ERR_POISONED: return "TQD_ERR_POISONED";
    case TQD_ERR_NOT_PREFILLED: return "TQD_ERR_NOT_PREFILLED";
    default: return "TQD_UNKNOWN_STATUS";
  }
}

const char* tqd_last_error(void) { return g_last_error.c_str(); }

void tqd_destroy(tqd_model* m) {
  if (!m) return;
  if (m->stream) cudaStreamSynchronize(m->stream);
  for (SeqSlot& s : m->seqs) {
    if (s.g_full) cudaGraphExecDestroy(s.g_full);
    if (s.g_layers) cudaGraphExecDestroy(s.g_layers);
  }
  for (auto& row : m->bgraph)
    for (cudaGraphExec_t& g : row)
    if (g) cudaGraphExecDestroy(g);
  for (auto& row : m->pgraph)
    for (cudaGraphExec_t& g : row)
      if (g) cudaGraphExecDestroy(g);
  if (m->arena) cudaFree(m->arena);
  if (m->h_tokens) cudaFreeHost(m->h_tokens);
  if (m->h_state) cudaFreeHost(m->h_state);
  if (m->own_stream && m->stream) cudaStreamDestroy(m->stream);
  delete m;
}

int32_t tqd_create(const tqd_config* cfg, const tqd_host_weights* w, void* stream,
                   tqd_model** out) {
  g_last_error.clear();
  if (!cfg || !w || !out) {
    set_error("cfg, weights and out must be non-NULL");
    return TQD_ERR_BAD_ARG;
  }
  *out = nullptr;
  int32_t rc = validate_config(cfg);
  if (rc) return rc;
  if ((rc = check_weights(cfg, w))) return rc;

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    set_error("no CUDA device");
    return TQD_ERR_NO_DEVICE;
  }
  tqd_model* m = new tqd_model();
  m->cfg = *cfg;
  m->stream = static_cast<cudaStream_t>(stream);
  cudaDeviceProp prop;
  cudaError_t pe = cudaGetDevice(&m->device);
  if (pe == cudaSuccess) pe = cudaGetDeviceProperties(&prop, m->device);
  if (pe != cudaSuccess) {
    set_error("device query failed: %s", cudaGetErrorString(pe));
    delete m;
    return TQD_ERR_CUDA;
  }
  if (prop.major * 10 + prop.minor != 103) {
    set_error("device %s is sm_%d%d; this library is built for sm_103a", prop.name, prop.major,
              prop.minor);
    delete m;
    return TQD_ERR_NO_DEVICE;
  }
  m->num_sms = prop.multiProcessorCount;
  if (!m->stream) {
    // the legacy default stream cannot be captured into a graph
    pe = cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking);
    if (pe != cudaSuccess) {
      set_error("stream creation failed: %s", cudaGetErrorString(pe));
      delete m;
      return TQD_ERR_CUDA;
    }
    m->own_stream = true;
  }
  if (const char* e = getenv("TQD_PDL")) m->pdl = atoi(e) != 0;

  const int L = cfg->n_layers, H = cfg->hidden, hd = cfg->head_dim, nq = cfg->n_heads,
            nkv = cfg->n_kv_heads, I = cfg->intermediate, V = cfg->vocab, S = cfg->max_seq;
  const int qw = nq * hd, kvw = nkv * hd, wt = cfg->weight_type;
  const int fmt = wt == TQD_WEIGHT_Q8_0 ? kFmtQ8 : kFmtBF16;
  const size_t rbh = row_bytes(wt, H), rbq = row_bytes(wt, qw), rbi = row_bytes(wt, I);
  // split-K attention chunks: one (kv head, chunk) item per SM, and few
  // enough that a group's partials (G x chunks x (head_dim + 2) floats) fit
  // the 24 KB the persistent kernel stages them in
  int nch = m->num_sms / nkv;
  const int nch_cap = 24576 / (4 * (nq / nkv) * (hd + 2));
  if (nch > nch_cap) nch = nch_cap;
  if (nch < 1) nch = 1;

  // ---- arena layout ----
  const size_t A = 256;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, A);
    return o;
  };
  // the persistent schedule reads wo's columns split by kv group: nkv
  // matrices [H x G hd], one per group
  const bool persist = cfg->schedule == TQD_SCHED_PERSISTENT;
  const int gh = (nq / nkv) * hd;
  const size_t rbg = row_bytes(wt, gh);
  // and the down projection by column blocks (DevModel::dcol_bytes)
  const size_t dcol = wt == TQD_WEIGHT_Q8_0 ? align_up(2ull * H, 16) + 32ull * H : 2ull * H;
  const size_t dcol_total = wt == TQD_WEIGHT_Q8_0 ? dcol * (I / 32) : dcol * I;
  struct LayerOff { size_t wqkv, wo, wog, wgu, wd, wdc, an, qn, kn, fn; };
  std::vector<LayerOff> lo(L);
  for (int l = 0; l < L; ++l) {
    lo[l].wqkv = take(rbh * (qw + 2 * kvw));
    lo[l].wo = take(rbq * H);
    lo[l].wog = persist ? take(rbg * H * nkv) : 0;
    lo[l].wgu = take(rbh * 2 * I);
    lo[l].wd = take(rbi * H);
    lo[l].wdc = persist ? take(dcol_total) : 0;
    lo[l].an = take(4 * H);
    lo[l].qn = take(4 * hd);
    lo[l].kn = take(4 * hd);
    lo[l].fn = take(4 * H);
  }
  const size_t o_lm = take(rbh * V);
  const size_t o_embed = w->embed ? take(rbh * V) : o_lm;
  const size_t o_onorm = take(4 * H);
  const size_t o_rope = take(sizeof(float2) * static_cast<size_t>(S) * (hd / 2));
  const size_t o_layers = take(sizeof(DevLayer) * L);
  const size_t weights_end = off;
  // the batched kernels' shapes (several sequences per step, prefill tiles, an f16 cache)
  DevModel shape{};
  shape.H = H; shape.nq = nq; shape.nkv = nkv; shape.hd = hd; shape.I = I; shape.qw = qw;
  const bool batched = batch_supported(shape) && (V + 127) / 128 <= kMaxArgmaxBlocks;
  const bool kv16 = cfg->kv_type == TQD_KV_F16;
  struct SeqOff { size_t state, tokens, kc, vc, x, xmid, qkv, attn, h, logits, po, pml, acnt, av, ai, acount, bar, gbar,
                  opart, sz, scnt, xacc, qkvt, sparts; };
  std::vector<SeqOff> so(cfg->max_batch);
  const size_t kv_bytes = (kv16 ? 2 : 4) * static_cast<size_t>(L) * S * kvw;
  for (int b = 0; b < cfg->max_batch; ++b) {
    so[b].state = take(sizeof(DevState));
    so[b].tokens = take(4 * (static_cast<size_t>(S) + 1));
    so[b].kc = take(kv_bytes);
    so[b].vc = take(kv_bytes);
    so[b].x = take(4 * H);
    so[b].xmid = take(4 * H);
    so[b].qkv = take(4 * (qw + 2 * kvw));
    so[b].attn = take(4 * qw);
    so[b].h = take(4 * I);
    so[b].logits = take(4 * align_up(static_cast<size_t>(V), 4));  // read as float4 groups by the sampler
    so[b].po = take(4 * static_cast<size_t>(nq) * nch * hd);
    so[b].pml = take(4 * static_cast<size_t>(nq) * nch * 2);
    so[b].acnt = take(4 * nkv);
    so[b].av = take(4 * kMaxArgmaxBlocks);
    so[b].ai = take(4 * kMaxArgmaxBlocks);
    so[b].acount = take(4);
    so[b].bar = take(sizeof(DevBarrier));
    so[b].gbar = take(sizeof(DevBarrier) * 16 * nkv);  // two per group, 128 bytes apart
    so[b].opart = take(4ull * 2 * H);  // the persistent schedule's O products, two sets
    so[b].sz = take(4 * align_up(static_cast<size_t>(V), 4));
    so[b].scnt = take(4 * align_up(static_cast<size_t>(V), 4));
    so[b].xacc = persist ? take(4ull * 2 * 4 * H) : 0;
    so[b].qkvt = persist ? take(8ull * (qw + 2 * kvw)) : 0;
    so[b].sparts = take(8ull * kSamplePartK * ((static_cast<size_t>(V) + kSampleSlice - 1) / kSampleSlice));
  }
  const size_t o_dseqs = take(sizeof(DevSeq) * cfg->max_batch);  // the descriptors, for kernels over sequences
  // batched-step buffers (several sequences per step, or a prompt's tiles),
  // for every shape the batched kernels support
  const int bmax = batch_max();
  size_t o_bx = 0, o_bqkv = 0, o_bpo = 0, o_bpml = 0, o_bh = 0, o_bcount = 0, o_bss = 0, o_blm = 0, o_bio = 0,
         o_pslots = 0, o_pstates = 0;
  if (batched) {
    o_bx = take(4ull * bmax * H);
    o_bqkv = take(4ull * bmax * (qw + 2 * kvw));
    o_bpo = take(4ull * bmax * nq * nch * hd);  // attention chunk partials (at most n_chunks chunks)
    o_bpml = take(4ull * bmax * nq * nch * 2);
    o_bh = take(4ull * bmax * I);
    o_bcount = take(4);
    o_bss = take(4ull * 2 * batch_ss_slots(H) * bmax);
    o_blm = take(batch_head_bytes(V, H, fmt));
    o_bio = take(4ull * 3 * 64);  // tokens in [64], argmaxes and error words out [2 x 64]
    o_pslots = take(sizeof(DevSeq) * (bmax + 1));
    o_pstates = take(sizeof(DevState) * bmax);
  }
  m->arena_bytes = off;
  cudaError_t ce = cudaMalloc(&m->arena, m->arena_bytes);
  if (ce != cudaSuccess) {
    cudaGetLastError();
    set_error("cudaMalloc of %zu bytes failed: %s", m->arena_bytes, cudaGetErrorString(ce));
    m->arena = nullptr;
    tqd_destroy(m);
    return TQD_ERR_OOM;
  }
  if (cudaMallocHost(&m->h_tokens, 4 * std::max<size_t>(static_cast<size_t>(S) + 1, 256)) != cudaSuccess ||
      cudaMallocHost(&m->h_state, sizeof(DevState)) != cudaSuccess) {
    cudaGetLastError();
    set_error("pinned host allocation failed");
    tqd_destroy(m);
    return TQD_ERR_OOM;
  }
  uint8_t* base = m->arena;
  cudaStream_t st = m->stream;
  auto fail = [&](cudaError_t e, const char* what) {
    int32_t r = fail_cuda(m, e, what);
    tqd_destroy(m);
    return r;
  };
  cudaError_t e = cudaMemsetAsync(base + weights_end, 0, m->arena_bytes - weights_end, st);
  if (e != cudaSuccess) return fail(e, "clear sequence state");

  // ---- weights: upload once, repack Q8_0 blocks into the row layout ----
  uint8_t* tmp = nullptr;
  if (wt == TQD_WEIGHT_Q8_0) {
    size_t maxm = host_row_bytes(wt, H) * static_cast<size_t>(V);
    size_t lm = host_row_bytes(wt, H) * (qw > 2 * I ? qw : 2 * I);
    if (lm > maxm) maxm = lm;
    if (host_row_bytes(wt, I) * H > maxm) maxm = host_row_bytes(wt, I) * H;
    if (host_row_bytes(wt, qw) * H > maxm) maxm = host_row_bytes(wt, qw) * H;
    ce = cudaMalloc(&tmp, maxm);
    if (ce != cudaSuccess) {
      cudaGetLastError();
      set_error("cudaMalloc of the upload buffer failed: %s", cudaGetErrorString(ce));
      tqd_destroy(m);
      return TQD_ERR_OOM;
    }
  }
  int64_t wbytes = 0;
  // upload `rows` x `cols` host rows to destination rows dst_row0 + r*step
  auto put = [&](const void* src, int rows, int cols, size_t dst_off, int dst_row0,
                 int step) -> cudaError_t {
    const size_t hrb = host_row_bytes(wt, cols), rb = row_bytes(wt, cols);
    wbytes += static_cast<int64_t>(rb) * rows;
    if (wt == TQD_WEIGHT_Q8_0) {
      cudaError_t r = cudaMemcpyAsync(tmp, src, hrb * rows, cudaMemcpyHostToDevice, st);
      if (r != cudaSuccess) return r;
      r = launch_q8_repack(tmp, rows, cols, base + dst_off, dst_row0, step, st);
      if (r != cudaSuccess) return r;
      return cudaStreamSynchronize(st);  // tmp is reused by the next upload
    }
    return cudaMemcpy2DAsync(base + dst_off + rb * dst_row0, rb * step, src, hrb, hrb, rows,
                             cudaMemcpyHostToDevice, st);
  };
  auto put_f32 = [&](const float* src, int n, size_t dst_off) -> cudaError_t {
    wbytes += 4ll * n;
    return cudaMemcpyAsync(base + dst_off, src, 4ull * n, cudaMemcpyHostToDevice, st);
  };
  std::vector<DevLayer> dl(L);
  for (int l = 0; l < L; ++l) {
    const tqd_layer_weights& W = w->layers[l];
    if ((e = put(W.wq, qw, H, lo[l].wqkv, 0, 1)) != cudaSuccess ||
        (e = put(W.wk, kvw, H, lo[l].wqkv, qw, 1)) != cudaSuccess ||
        (e = put(W.wv, kvw, H, lo[l].wqkv, qw + kvw, 1)) != cudaSuccess ||
        (e = put(W.wo, H, qw, lo[l].wo, 0, 1)) != cudaSuccess ||
        (e = put(W.w_gate, I, H, lo[l].wgu, 0, 2)) != cudaSuccess ||
        (e = put(W.w_up, I, H, lo[l].wgu, 1, 2)) != cudaSuccess ||
        (e = put(W.w_down, H, I, lo[l].wd, 0, 1)) != cudaSuccess ||
        (e = put_f32(W.attn_norm, H, lo[l].an)) != cudaSuccess ||
        (e = put_f32(W.ffn_norm, H, lo[l].fn)) != cudaSuccess) {
      if (tmp) cudaFree(tmp);
      return fail(e, "upload layer weights");
    }
    if (cfg->qk_norm && ((e = put_f32(W.q_norm, hd, lo[l].qn)) != cudaSuccess ||
                         (e = put_f32(W.k_norm, hd, lo[l].kn)) != cudaSuccess)) {
      if (tmp) cudaFree(tmp);
      return fail(e, "upload qk-norm gains");
    }
    if (persist) {
      // wo's columns of each kv group as its own [H x gh] matrix
      const size_t hrb = host_row_bytes(wt, qw), hsb = host_row_bytes(wt, gh);
      std::vector<uint8_t> slice(hsb * H);
      for (int g = 0; g < nkv && e == cudaSuccess; ++g) {
        const uint8_t* src = static_cast<const uint8_t*>(W.wo);
        for (int r = 0; r < H; ++r)
          memcpy(slice.data() + hsb * r, src + hrb * r + hsb * g, hsb);
        e = put(slice.data(), H, gh, lo[l].wog + rbg * H * g, 0, 1);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);  // the host slice is reused
        wbytes -= static_cast<int64_t>(rbg) * H;  // a second layout of wo, not more weights
      }
      if (e != cudaSuccess) {
        if (tmp) cudaFree(tmp);
        return fail(e, "upload the grouped O projection");
      }
      dl[l].wo_g = base + lo[l].wog;
      // wd by column blocks: the block a CTA streams holds exactly the columns
      // that multiply the SwiGLU outputs it computed
      std::vector<uint8_t> cols(dcol_total);
      const uint8_t* src = static_cast<const uint8_t*>(W.w_down);
      const size_t hrb_d = host_row_bytes(wt, I);
      if (wt == TQD_WEIGHT_Q8_0) {
        for (int c = 0; c < I / 32; ++c) {
          uint8_t* blk = cols.data() + dcol * c;
          uint8_t* q = blk + align_up(2ull * H, 16);
          for (int r = 0; r < H; ++r) {
            const uint8_t* b34 = src + hrb_d * r + 34ull * c;
            blk[2 * r] = b34[0];
            blk[2 * r + 1] = b34[1];
            for (int j = 0; j < 32; ++j) q[static_cast<size_t>(j) * H + r] = b34[2 + j];
          }
        }
      } else {
        uint16_t* dst16 = reinterpret_cast<uint16_t*>(cols.data());
        for (int r = 0; r < H; ++r) {
          const uint8_t* row = src + hrb_d * r;
          for (int j = 0; j < I; ++j) {
            uint16_t v;
            memcpy(&v, row + 2ull * j, 2);
            dst16[static_cast<size_t>(j) * H + r] = v;
          }
        }
      }
      e = cudaMemcpyAsync(base + lo[l].wdc, cols.data(), dcol_total, cudaMemcpyHostToDevice, st);
      if (e == cudaSuccess) e = cudaStreamSynchronize(st);  // the host copy is freed below
      if (e != cudaSuccess) {
        if (tmp) cudaFree(tmp);
        return fail(e, "upload the down projection by columns");
      }
      dl[l].wd_c = base + lo[l].wdc;
    }
    dl[l].wqkv = base + lo[l].wqkv;
    dl[l].wo = base + lo[l].wo;
    dl[l].wgu = base + lo[l].wgu;
    dl[l].wd = base + lo[l].wd;
    dl[l].attn_norm = reinterpret_cast<const float*>(base + lo[l].an);
    dl[l].q_norm = reinterpret_cast<const float*>(base + lo[l].qn);
    dl[l].k_norm = reinterpret_cast<const float*>(base + lo[l].kn);
    dl[l].ffn_norm = reinterpret_cast<const float*>(base + lo[l].fn);
  }
  if ((e = put(w->lm_head, V, H, o_lm, 0, 1)) != cudaSuccess ||
      (w->embed && (e = put(w->embed, V, H, o_embed, 0, 1)) != cudaSuccess) ||
      (e = put_f32(w->out_norm, H, o_onorm)) != cudaSuccess ||
      (e = cudaMemcpyAsync(base + o_layers, dl.data(), sizeof(DevLayer) * L,
                           cudaMemcpyHostToDevice, st)) != cudaSuccess ||
      (e = launch_rope_table(static_cast<double>(cfg->rope_theta), hd, S,
                             reinterpret_cast<float2*>(base + o_rope), st)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess) {
    if (tmp) cudaFree(tmp);
    return fail(e, "upload head weights");
  }
  if (batched &&
      ((e = launch_head_tile(base + o_lm, rbh, V, H, fmt, base + o_blm, st)) != cudaSuccess ||
       (e = cudaStreamSynchronize(st)) != cudaSuccess)) {
    if (tmp) cudaFree(tmp);
    return fail(e, "tile the lm_head");
  }
  if (tmp) cudaFree(tmp);
  m->host_layers = dl;
  if (w->embed) wbytes -= static_cast<int64_t>(row_bytes(wt, H)) * V;  // one row per step
  m->weight_bytes = wbytes;

  DevModel& dm = m->dm;
  dm.n_layers = L; dm.H = H; dm.nq = nq; dm.nkv = nkv; dm.hd = hd; dm.I = I; dm.V = V;
  dm.qk_norm = cfg->qk_norm; dm.wtype = fmt; dm.max_seq = S;
  dm.qw = qw; dm.kvw = kvw; dm.n_chunks = nch;
  dm.eps = cfg->rms_eps;
  dm.attn_scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(hd)));
  dm.row_bytes_h = rbh; dm.row_bytes_qw = rbq; dm.row_bytes_i = rbi; dm.row_bytes_gh = rbg;
  dm.dcol_bytes = dcol;
  dm.layers = reinterpret_cast<const DevLayer*>(base + o_layers);
  dm.lm_head = base + o_lm;
  dm.embed = base + o_embed;
  dm.out_norm = reinterpret_cast<const float*>(base + o_onorm);
  dm.rope = reinterpret_cast<const float2*>(base + o_rope);
  dm.kv16 = kv16 ? 1 : 0;

  m->seqs.resize(cfg->max_batch);
  for (int b = 0; b < cfg->max_batch; ++b) {
    DevSeq& d = m->seqs[b].d;
    d.state = reinterpret_cast<DevState*>(base + so[b].state);
    d.tokens = reinterpret_cast<int32_t*>(base + so[b].tokens);
    d.kcache = reinterpret_cast<float*>(base + so[b].kc);
    d.vcache = reinterpret_cast<float*>(base + so[b].vc);
    d.x = reinterpret_cast<float*>(base + so[b].x);
    d.x_mid = reinterpret_cast<float*>(base + so[b].xmid);
    d.qkv = reinterpret_cast<float*>(base + so[b].qkv);
    d.attn = reinterpret_cast<float*>(base + so[b].attn);
    d.h = reinterpret_cast<float*>(base + so[b].h);
    d.logits = reinterpret_cast<float*>(base + so[b].logits);
    d.part_o = reinterpret_cast<float*>(base + so[b].po);
    d.part_ml = reinterpret_cast<float*>(base + so[b].pml);
    d.attn_count = reinterpret_cast<uint32_t*>(base + so[b].acnt);
    d.amax_v = reinterpret_cast<float*>(base + so[b].av);
    d.amax_i = reinterpret_cast<int32_t*>(base + so[b].ai);
    d.amax_count = reinterpret_cast<uint32_t*>(base + so[b].acount);
    d.bar = reinterpret_cast<DevBarrier*>(base + so[b].bar);
    d.gbar = reinterpret_cast<DevBarrier*>(base + so[b].gbar);
    d.opart = reinterpret_cast<float*>(base + so[b].opart);
    d.sz = reinterpret_cast<float*>(base + so[b].sz);
    d.scnt = reinterpret_cast<uint32_t*>(base + so[b].scnt);
    d.xacc = persist ? reinterpret_cast<float*>(base + so[b].xacc) : nullptr;
    d.qkv_tag = persist ? reinterpret_cast<uint64_t*>(base + so[b].qkvt) : nullptr;
    d.sparts = reinterpret_cast<unsigned long long*>(base + so[b].sparts);
    d.tok_in = -1;
  }
  m->dseqs = reinterpret_cast<DevSeq*>(base + o_dseqs);
  {
    std::vector<DevSeq> hs(cfg->max_batch);
    for (int b = 0; b < cfg->max_batch; ++b) hs[b] = m->seqs[b].d;
    if ((e = cudaMemcpy(m->dseqs, hs.data(), sizeof(DevSeq) * cfg->max_batch, cudaMemcpyHostToDevice)) !=
        cudaSuccess)
      return fail(e, "upload sequence descriptors");
  }
  if (batched) {
    m->bx = reinterpret_cast<float*>(base + o_bx);
    m->bqkv = reinterpret_cast<float*>(base + o_bqkv);
    m->bpo = reinterpret_cast<float*>(base + o_bpo);
    m->bpml = reinterpret_cast<float*>(base + o_bpml);
    m->bh = reinterpret_cast<float*>(base + o_bh);
    m->bcount = reinterpret_cast<uint32_t*>(base + o_bcount);
    m->bss = reinterpret_cast<float*>(base + o_bss);
    m->blm = base + o_blm;
    m->bio = reinterpret_cast<int32_t*>(base + o_bio);
    m->pslots = reinterpret_cast<DevSeq*>(base + o_pslots);
    m->pstates = reinterpret_cast<DevState*>(base + o_pstates);
    if ((e = batch_setup(dm)) != cudaSuccess) return fail(e, "batched-step set-up");
    m->batch_ok = true;
  }
  m->blocks_qkv = matvec_blocks(fmt, qw + 2 * kvw, H, m->num_sms, 0);
  m->blocks_o = matvec_blocks(fmt, H, qw, m->num_sms, 0);
  m->blocks_gu = matvec_blocks(fmt, 2 * I, H, m->num_sms, 0);
  m->blocks_d = matvec_blocks(fmt, H, I, m->num_sms, 0);
  m->blocks_lm = matvec_blocks(fmt, V, H, m->num_sms, kMaxArgmaxBlocks);
  if (cfg->schedule == TQD_SCHED_PERSISTENT) {
    const int per_sm = persistent_blocks_per_sm(m->dm);
    if (per_sm < 1) {
      cudaGetLastError();
      set_error("persistent kernel cannot be resident on an SM (%zu bytes of shared memory)",
                persistent_smem_bytes(m->dm));
      tqd_destroy(m);
      return TQD_ERR_UNSUPPORTED_CONFIG;
    }
    m->blocks_persist = m->num_sms;
  }
  *out = m;
  return TQD_OK;
}

int32_t tqd_reset(tqd_model* m, int32_t seq) {
  int32_t rc = check_model(m, seq);
  if (rc) return rc;
  SeqSlot& s = m->seqs[seq];
  CK(cudaMemsetAsync(s.d.state, 0, sizeof(DevState), m->stream), "reset state");
  CK(cudaStreamSynchronize(m->stream), "synchronize");
  s.next_pos = 0;
  s.logits_pos = -1;
  return TQD_OK;
}

int32_t tqd_truncate(tqd_model* m, int32_t seq, int32_t n_pos) {
  int32_t rc = check_model(m, seq);
  if (rc) return rc;
  SeqSlot& s = m->seqs[seq];
  if (n_pos < 0 || n_pos > s.next_pos) {
    set_error("truncate to %d outside [0, %d]", n_pos, s.next_pos);
    return TQD_ERR_BAD_ARG;
  }
  DevState st{};
  st.pos = static_cast<uint32_t>(n_pos);
  *m->h_state = st;
  CK(cudaMemcpyAsync(s.d.state, m->h_state, sizeof(DevState), cudaMemcpyHostToDevice, m->stream),
     "set position");
  CK(cudaStreamSynchronize(m->stream), "synchronize");
  if (n_pos != s.next_pos) s.logits_pos = -1;
  s.next_pos = n_pos;
  return TQD_OK;
}

int32_t tqd_next_pos(tqd_model* m, int32_t seq, int32_t* pos_out) {
  int32_t rc = check_model(m, seq);
  if (rc) return rc;
  if (!pos_out) {
    set_error("pos_out is NULL");
    return TQD_ERR_BAD_ARG;
  }
  *pos_out = m->seqs[seq].next_pos;
  return TQD_OK;
}

int32_t tqd_prefill(tqd_model* m, int32_t seq, const int32_t* ids, int32_t n, int32_t* next_out) {
  int32_t rc = check_model(m, seq);
  if (rc) return rc;
  if (!ids || !next_out || n <= 0) {
    set_error("prefill needs ids, next_out and n > 0");
    return TQD_ERR_BAD_ARG;
  }
  SeqSlot& s = m->seqs[seq];
  const int32_t pos = s.next_pos;
  if (static_cast<int64_t>(pos) + n > m->cfg.max_seq) {
    set_error("prefill of %d tokens at position %d exceeds max_seq %d", n, pos, m->cfg.max_seq);
    return TQD_ERR_CAPACITY;
  }
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= m->cfg.vocab) {
      set_error("token id %d at index %d outside the vocabulary", ids[i], i);
      return TQD_ERR_BAD_ARG;
    }
  memcpy(m->h_tokens, ids, 4ull * n);
  CK(cudaMemcpyAsync(s.d.tokens + pos, m->h_tokens, 4ull * n, cudaMemcpyHostToDevice, m->stream),
     "upload prompt");
  if ((rc = run_steps(m, s, n, n - 1))) return rc;
  CK(cudaMemcpyAsync(m->h_tokens, s.d.tokens + pos + n, 4, cudaMemcpyDeviceToHost, m->stream),
     "read next token");
  if ((rc = finish(m, s))) return rc;
  s.next_pos = pos + n;
  s.logits_pos = s.next_pos;
  *next_out = m->h_tokens[0];
  return TQD_OK;
}

int32_t tqd_kv_upload(tqd_model* m, int32_t seq, int32_t n_pos, const float* k, const float* v) {
  int32_t rc = check_model(m, seq);
  if (rc) return rc;
  if (!k || !v || n_pos < 0) {
    set_error("kv_upload needs k, v and n_pos >= 0");
    return TQD_ERR_BAD_ARG;
  }
  if (n_pos > m->cfg.max_seq) {
    set_error("n_pos %d exceeds max_seq %d", n_pos, m->cfg.max_seq);
    return TQD_ERR_CAPACITY;
  }
  SeqSlot& s = m->seqs[seq];
  const size_t kvw = static_cast<size_t>(m->dm.kvw);
  if (n_pos > 0) {
    // host rows [layer][pos][kv head * head_dim] -> device [layer][kv head][pos][head_dim];
    // an f16 cache takes the rows rounded to nearest-even binary16
    const size_t hd = static_cast<size_t>(m->dm.hd), es = m->dm.kv16 ? 2 : 4;
    std::vector<__half> k16, v16;
    const uint8_t* ksrc = reinterpret_cast<const uint8_t*>(k);
    const uint8_t* vsrc = reinterpret_cast<const uint8_t*>(v);
    if (m->dm.kv16) {
      const size_t n = static_cast<size_t>(m->cfg.n_layers) * n_pos * kvw;
      k16.resize(n);
      v16.resize(n);
      for (size_t i = 0; i < n; ++i) {
        k16[i] = __float2half_rn(k[i]);
        v16[i] = __float2half_rn(v[i]);
      }
      ksrc = reinterpret_cast<const uint8_t*>(k16.data());
      vsrc = reinterpret_cast<const uint8_t*>(v16.data());
    }
    uint8_t* kdev = reinterpret_cast<uint8_t*>(s.d.kcache);
    uint8_t* vdev = reinterpret_cast<uint8_t*>(s.d.vcache);
    for (int l = 0; l < m->cfg.n_layers; ++l)
      for (int g = 0; g < m->dm.nkv; ++g) {
        const size_t src = (static_cast<size_t>(l) * n_pos) * kvw + g * hd;
        const size_t dst = (static_cast<size_t>(l) * m->dm.nkv + g) * m->cfg.max_seq * hd;
        CK(cudaMemcpy2DAsync(kdev + dst * es, es * hd, ksrc + src * es, es * kvw, es * hd, n_pos,
                             cudaMemcpyHostToDevice, m->stream),
           "upload K");
        CK(cudaMemcpy2DAsync(vdev + dst * es, es * hd, vsrc + src * es, es * kvw, es * hd, n_pos,
                             cudaMemcpyHostToDevice, m->stream),
           "upload V");
      }
    CK(cudaStreamSynchronize(m->stream), "synchronize");  // the converted rows are copied
  }
  DevState st{};
  st.pos = static_cast<uint32_t>(n_pos);
  *m->h_state = st;
  CK(cudaMemcpyAsync(s.d.state, m->h_state, sizeof(DevState), cudaMemcpyHostToDevice, m->stream),
     "set position");
  CK(cudaStreamSynchronize(m->stream), "synchronize");
  s.next_pos = n_pos;
  s.logits_pos = -1;
  return TQD_OK;
}

int32_t tqd_decode_step(tqd_model* m, int32_t seq, int32_t token, int32_t pos, int32_t* next_out) {
  int32_t rc = check_model(m, seq);
  if (rc) return rc;
  if (!next_out || token < 0 || token >= m->cfg.vocab) {
    set_error("decode_step needs next_out and a token in [0, vocab)");
    return TQD_ERR_BAD_ARG;
  }
  SeqSlot& s = m->seqs[seq];
  if (pos != s.next_pos) {
    set_error("pos %d is not the sequence's next position %d", pos, s.next_pos);
    return TQD_ERR_POS_MISMATCH;
  }
  if (pos >= m->cfg.max_seq) {
    set_error("position %d is beyond max_seq %d", pos, m->cfg.max_seq);
    return TQD_ERR_CAPACITY;
  }
  if (m->cfg.schedule == TQD_SCHED_PERSISTENT) {
    // the token goes in as a launch argument and the next one comes back in
    // the state record finish() reads: one launch and one readback per token
    DevSeq d = s.d;
    d.tok_in = token;
    CK(launch_persistent(m->dm, d, 1, 0, m->blocks_persist, m->stream), "persistent launch");
  } else {
    m->h_tokens[0] = token;
    CK(cudaMemcpyAsync(s.d.tokens + pos, m->h_tokens, 4, cudaMemcpyHostToDevice, m->stream),
       "write token");
    if ((rc = run_steps(m, s, 1, 0))) return rc;
  }
  if ((rc = finish(m, s))) return rc;
  s.next_pos = pos + 1;
  s.logits_pos = s.next_pos;
  *next_out = m->h_state->last;
  return TQD_OK;
}

namespace {

// Check the caller's sampling controls and turn them into kernel arguments;
// *greedy when the temperature asks for the argmax.
int32_t sample_args(const tqd_sampling* p, SampleArgs& a, bool* greedy) {
  if (!p) {
    set_error("sampling controls are NULL");
    return TQD_ERR_BAD_ARG;
  }
  if (!std::isfinite(p->temperature) || !std::isfinite(p->top_p) || !std::isfinite(p->min_p) ||
      !std::isfinite(p->repeat_penalty) || !std::isfinite(p->presence_penalty) ||
      !std::isfinite(p->frequency_penalty)) {
    set_error("sampling controls must be finite");
    return TQD_ERR_BAD_ARG;
  }
  if (p->top_k < 0 || !(p->top_p > 0.f) || p->top_p > 1.f || p->min_p < 0.f || p->min_p > 1.f ||
      !(p->repeat_penalty > 0.f)) {
    set_error("sampling controls out of range: top_k >= 0, top_p in (0, 1], min_p in [0, 1], repeat_penalty > 0");
    return TQD_ERR_BAD_ARG;
  }
  *greedy = p->temperature <= 0.f;
  a.temperature = p->temperature;
  a.top_k = p->top_k;
  a.top_p = p->top_p;
  a.ln_min_p = p->min_p > 0.f ? static_cast<float>(std::log(static_cast<double>(p->min_p))) : -INFINITY;
  a.repeat = p->repeat_penalty;
  a.presence = p->presence_penalty;
  a.frequency = p->frequency_penalty;
  a.penalize = p->repeat_penalty != 1.f || p->presence_penalty != 0.f || p->frequency_penalty != 0.f;
  a.seed = p->seed;
  return TQD_OK;
}

// n_steps device-chained steps of one sequence; with sa, each step's token is
// drawn by the sampler instead of the argmax.
int32_t generate_impl(tqd_model* m, int32_t seq, int32_t first_token, int32_t n_steps, int32_t* ids_out,
                      const SampleArgs* sa) {
  int32_t rc = check_model(m, seq);
  if (rc) return rc;
  if (!ids_out || n_steps <= 0 || first_token < 0 || first_token >= m->cfg.vocab) {
    set_error("generate needs ids_out, n_steps > 0 and a first token in [0, vocab)");
    return TQD_ERR_BAD_ARG;
  }
  SeqSlot& s = m->seqs[seq];
  const int32_t pos = s.next_pos;
  if (static_cast<int64_t>(pos) + n_steps > m->cfg.max_seq) {
    set_error("%d steps at position %d exceed max_seq %d", n_steps, pos, m->cfg.max_seq);
    return TQD_ERR_CAPACITY;
  }
  m->h_tokens[0] = first_token;
  CK(cudaMemcpyAsync(s.d.tokens + pos, m->h_tokens, 4, cudaMemcpyHostToDevice, m->stream),
     "write token");
  if (!sa) {
    if ((rc = run_steps(m, s, n_steps, 0))) return rc;
  } else {
    for (int i = 0; i < n_steps; ++i) {
      if ((rc = run_steps(m, s, 1, 0))) return rc;
      CK(launch_sample(m->dseqs + seq, 1, m->cfg.vocab, m->cfg.max_seq, *sa, m->stream, true), "sampler launch");
    }
  }
  CK(cudaMemcpyAsync(m->h_tokens, s.d.tokens + pos + 1, 4ull * n_steps, cudaMemcpyDeviceToHost,
                     m->stream),
     "read tokens");
  if ((rc = finish(m, s))) return rc;
  s.next_pos = pos + n_steps;
  s.logits_pos = s.next_pos;
  memcpy(ids_out, m->h_tokens, 4ull * n_steps);
  return TQD_OK;
}

}  // namespace

extern "C++" {
namespace tqd {
int32_t sampling_args(const tqd_sampling* p, SampleArgs& a, bool* greedy) { return sample_args(p, a, greedy); }
}  // namespace tqd
}

int32_t tqd_generate(tqd_model* m, int32_t seq, int32_t first_token, int32_t n_steps, int32_t* ids_out) {
  return generate_impl(m, seq, first_token, n_steps, ids_out, nullptr);
}

int32_t tqd_generate_sampled(tqd_model* m, int32_t seq, int32_t first_token, int32_t n_steps,
                             const tqd_sampling* sampling, int32_t* ids_out) {
  SampleArgs a{};
  bool greedy = false;
  const int32_t rc = sample_args(sampling, a, &greedy);
  if (rc) return rc;
  return generate_impl(m, seq, first_token, n_steps, ids_out, greedy ? nullptr : &a);
}

int32_t tqd_sample(tqd_model* m, int32_t seq, const tqd_sampling* sampling, int32_t* token_out) {
  int32_t rc = check_model(m, seq);
  if (rc) return rc;
  SampleArgs a{};
  bool greedy = false;
  if ((rc = sample_args(sampling, a, &greedy))) return rc;
  if (greedy) a.temperature = 0.f;
  if (!token_out) {
    set_error("token_out is NULL");
    return TQD_ERR_BAD_ARG;
  }
  SeqSlot& s = m->seqs[seq];
  if (s.next_pos == 0 || s.logits_pos != s.next_pos) {
    set_error("sequence %d has no logits for its next position %d: run a prefill or a step first", seq,
              s.next_pos);
    return TQD_ERR_NOT_PREFILLED;
  }
  // (greedy too: an earlier draw may have replaced the step's argmax at this position)
  CK(launch_sample(m->dseqs + seq, 1, m->cfg.vocab, m->cfg.max_seq, a, m->stream, true), "sampler launch");
  CK(cudaMemcpyAsync(m->h_tokens, s.d.tokens + s.next_pos, 4, cudaMemcpyDeviceToHost, m->stream), "read token");
  if ((rc = finish(m, s))) return rc;
  *token_out = m->h_tokens[0];
  return TQD_OK;
}

namespace {

int32_t check_batch(tqd_model* m, int32_t n_seq) {
  int32_t rc = check_model(m, 0);
  if (rc) return rc;
  if (!m->batch_ok || (m->cfg.max_batch < 2 && m->cfg.kv_type != TQD_KV_F16)) {
    set_error("this model has no batched step (max_batch must be > 1 and the shape supported)");
    return TQD_ERR_UNSUPPORTED_CONFIG;
  }
  if (n_seq < 1 || n_seq > m->cfg.max_batch) {
    set_error("n_seq %d outside [1, %d]", n_seq, m->cfg.max_batch);
    return TQD_ERR_BAD_ARG;
  }
  return TQD_OK;
}

// Enqueue `steps` batched steps of sequences 0..n-1: consecutive groups of at
// most batch_max() sequences, each one sweep of the weights (one graph per
// group and size, captured on first use).
int32_t run_batch(tqd_model* m, int n, int steps) {
  const int bm = batch_max(), groups = (n + bm - 1) / bm;
  for (int gi = 0; gi < groups; ++gi) {
    const int ng = std::min(bm, n - gi * bm);
    cudaGraphExec_t& g = m->bgraph[gi][ng];
    if (g) continue;
    // split-K chunks: as many as keep every (sequence, kv head, chunk) block
    // in one wave at two blocks per SM (a partial last wave would run alone)
    int nch = 2 * m->num_sms / (ng * m->dm.nkv);
    if (nch > m->dm.n_chunks) nch = m->dm.n_chunks;
    if (nch < 1) nch = 1;
    cudaGraph_t graph = nullptr;
    CK(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal), "begin capture");
    cudaError_t e = enqueue_batch_step(m->dm, m->host_layers.data(), m->blm, m->dseqs + gi * bm, ng, nch, m->bx,
                                       m->bqkv, m->bpo, m->bpml, m->bh, m->bss, m->bcount,
                                       &m->seqs[gi * bm].d.state->err, m->stream, false, 0);
    cudaError_t e2 = cudaStreamEndCapture(m->stream, &graph);
    if (e != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      return fail_cuda(m, e, "capture batched step");
    }
    if (e2 != cudaSuccess) return fail_cuda(m, e2, "end capture");
    e = cudaGraphInstantiate(&g, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return fail_cuda(m, e, "instantiate batched graph");
  }
  for (int i = 0; i < steps; ++i)
    for (int gi = 0; gi < groups; ++gi)
      CK(cudaGraphLaunch(m->bgraph[gi][std::min(bm, n - gi * bm)], m->stream), "batched graph launch");
  return TQD_OK;
}

// Enqueue one prefill tile of n positions for the sequence in m->pslots:
// slot positions, the batched step in tile mode (the lm_head on the last
// slot only where the tile ends the prompt), the sequence's advance.  One
// graph per (n, last).
int32_t run_prefill_tile(tqd_model* m, int n, bool last) {
  cudaGraphExec_t& g = m->pgraph[n][last ? 1 : 0];
  if (!g) {
    int nch = 2 * m->num_sms / (n * m->dm.nkv);
    if (nch > m->dm.n_chunks) nch = m->dm.n_chunks;
    if (nch < 1) nch = 1;
    cudaGraph_t graph = nullptr;
    CK(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal), "begin capture");
    cudaError_t e = launch_prefill_tile_begin(m->pslots, n, m->stream);
    if (e == cudaSuccess)
      e = enqueue_batch_step(m->dm, m->host_layers.data(), m->blm, m->pslots, n, nch, m->bx, m->bqkv, m->bpo,
                             m->bpml, m->bh, m->bss, m->bcount, &m->pstates[0].err, m->stream, true,
                             last ? n - 1 : n);
    if (e == cudaSuccess) e = launch_prefill_tile_end(m->pslots, n, m->stream);
    cudaError_t e2 = cudaStreamEndCapture(m->stream, &graph);
    if (e != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      return fail_cuda(m, e, "capture prefill tile");
    }
    if (e2 != cudaSuccess) return fail_cuda(m, e2, "end capture");
    e = cudaGraphInstantiate(&g, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return fail_cuda(m, e, "instantiate prefill tile");
  }
  CK(cudaGraphLaunch(g, m->stream), "prefill tile launch");
  return TQD_OK;
}

// Read back every sequence's state; the first error wins.
int32_t finish_batch(tqd_model* m, int n) {
  int32_t first = TQD_OK;
  for (int b = 0; b < n; ++b) {
    int32_t rc = finish(m, m->seqs[b]);
    if (rc && !first) first = rc;
    if (rc == TQD_ERR_DEVICE_TIMEOUT || rc == TQD_ERR_CUDA) return rc;
  }
  return first;
}

}  // namespace

int32_t tqd_decode_step_batch(tqd_model* m, int32_t n_seq, const int32_t* tokens, const int32_t* pos,
                              int32_t* next_out) {
  int32_t rc = check_batch(m, n_seq);
  if (rc) return rc;
  if (!tokens || !pos || !next_out) {
    set_error("tokens, pos and next_out must be non-NULL");
    return TQD_ERR_BAD_ARG;
  }
  for (int b = 0; b < n_seq; ++b) {
    if (tokens[b] < 0 || tokens[b] >= m->cfg.vocab) {
      set_error("token %d of sequence %d outside the vocabulary", tokens[b], b);
      return TQD_ERR_BAD_ARG;
    }
    if (pos[b] != m->seqs[b].next_pos) {
      set_error("pos %d of sequence %d is not its next position %d", pos[b], b, m->seqs[b].next_pos);
      return TQD_ERR_POS_MISMATCH;
    }
    if (pos[b] >= m->cfg.max_seq) {
      set_error("position %d of sequence %d is beyond max_seq %d", pos[b], b, m->cfg.max_seq);
      return TQD_ERR_CAPACITY;
    }
  }
  // one upload of the tokens, the step, one readback of the argmaxes and error words
  memcpy(m->h_tokens, tokens, 4ull * n_seq);
  CK(cudaMemcpyAsync(m->bio, m->h_tokens, 4ull * n_seq, cudaMemcpyHostToDevice, m->stream), "write tokens");
  CK(launch_batch_tokens_in(m->dseqs, n_seq, m->bio, m->stream), "place tokens");
  if ((rc = run_batch(m, n_seq, 1))) return rc;
  CK(launch_batch_tokens_out(m->dseqs, n_seq, m->bio + 64, m->stream), "gather tokens");
  CK(cudaMemcpyAsync(m->h_tokens + 64, m->bio + 64, 8ull * n_seq, cudaMemcpyDeviceToHost, m->stream),
     "read next tokens");
  CK(cudaStreamSynchronize(m->stream), "synchronize");
  for (int b = 0; b < n_seq; ++b)
    if (m->h_tokens[64 + n_seq + b] != 0) return finish_batch(m, n_seq);  // reports and clears the error
  for (int b = 0; b < n_seq; ++b) {
    m->seqs[b].next_pos = pos[b] + 1;
    m->seqs[b].logits_pos = m->seqs[b].next_pos;
    next_out[b] = m->h_tokens[64 + b];
  }
  return TQD_OK;
}

namespace {

int32_t generate_batch_impl(tqd_model* m, int32_t n_seq, const int32_t* first_tokens, int32_t n_steps,
                            int32_t* ids_out, const SampleArgs* sa) {
  int32_t rc = check_batch(m, n_seq);
  if (rc) return rc;
  if (!first_tokens || !ids_out || n_steps <= 0) {
    set_error("generate_batch needs first_tokens, ids_out and n_steps > 0");
    return TQD_ERR_BAD_ARG;
  }
  for (int b = 0; b < n_seq; ++b) {
    if (first_tokens[b] < 0 || first_tokens[b] >= m->cfg.vocab) {
      set_error("first token of sequence %d outside the vocabulary", b);
      return TQD_ERR_BAD_ARG;
    }
    if (static_cast<int64_t>(m->seqs[b].next_pos) + n_steps > m->cfg.max_seq) {
      set_error("%d steps from position %d of sequence %d exceed max_seq %d", n_steps,
                m->seqs[b].next_pos, b, m->cfg.max_seq);
      return TQD_ERR_CAPACITY;
    }
  }
  for (int b = 0; b < n_seq; ++b) {
    m->h_tokens[b] = first_tokens[b];
    CK(cudaMemcpyAsync(m->seqs[b].d.tokens + m->seqs[b].next_pos, m->h_tokens + b, 4,
                       cudaMemcpyHostToDevice, m->stream),
       "write token");
  }
  if (!sa) {
    if ((rc = run_batch(m, n_seq, n_steps))) return rc;
  } else {
    for (int i = 0; i < n_steps; ++i) {
      if ((rc = run_batch(m, n_seq, 1))) return rc;
      CK(launch_sample(m->dseqs, n_seq, m->cfg.vocab, m->cfg.max_seq, *sa, m->stream, true), "sampler launch");
    }
  }
  CK(cudaStreamSynchronize(m->stream), "synchronize");
  for (int b = 0; b < n_seq; ++b) {
    CK(cudaMemcpyAsync(m->h_tokens, m->seqs[b].d.tokens + m->seqs[b].next_pos + 1, 4ull * n_steps,
                       cudaMemcpyDeviceToHost, m->stream),
       "read tokens");
    CK(cudaStreamSynchronize(m->stream), "synchronize");
    for (int i = 0; i < n_steps; ++i) ids_out[static_cast<size_t>(i) * n_seq + b] = m->h_tokens[i];
  }
  if ((rc = finish_batch(m, n_seq))) return rc;
  for (int b = 0; b < n_seq; ++b) {
    m->seqs[b].next_pos += n_steps;
    m->seqs[b].logits_pos = m->seqs[b].next_pos;
  }
  return TQD_OK;
}

}  // namespace

int32_t tqd_generate_batch(tqd_model* m, int32_t n_seq, const int32_t* first_tokens, int32_t n_steps,
                           int32_t* ids_out) {
  return generate_batch_impl(m, n_seq, first_tokens, n_steps, ids_out, nullptr);
}

int32_t tqd_generate_batch_sampled(tqd_model* m, int32_t n_seq, const int32_t* first_tokens, int32_t n_steps,
                                   const tqd_sampling* sampling, int32_t* ids_out) {
  SampleArgs a{};
  bool greedy = false;
  const int32_t rc = sample_args(sampling, a, &greedy);
  if (rc) return rc;
  return generate_batch_impl(m, n_seq, first_tokens, n_steps, ids_out, greedy ? nullptr : &a);
}

int32_t tqd_prefill_batch(tqd_model* m, int32_t seq, const int32_t* ids, int32_t n, int32_t* next_out) {
  int32_t rc = check_model(m, seq);
  if (rc) return rc;
  if (!m->batch_ok) {
    set_error("this model's shape has no batched step, so no prefill tiles");
    return TQD_ERR_UNSUPPORTED_CONFIG;
  }
  if (!ids || !next_out || n <= 0) {
    set_error("prefill_batch needs ids, next_out and n > 0");
    return TQD_ERR_BAD_ARG;
  }
  SeqSlot& s = m->seqs[seq];
  const int32_t pos = s.next_pos;
  if (static_cast<int64_t>(pos) + n > m->cfg.max_seq) {
    set_error("prefill of %d tokens at position %d exceeds max_seq %d", n, pos, m->cfg.max_seq);
    return TQD_ERR_CAPACITY;
  }
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= m->cfg.vocab) {
      set_error("token id %d at index %d outside the vocabulary", ids[i], i);
      return TQD_ERR_BAD_ARG;
    }
  const int bmax = batch_max();
  // the tile slots: the sequence's descriptor with a state word of their own
  m->pslots_host.assign(bmax + 1, s.d);
  for (int b = 0; b < bmax; ++b) m->pslots_host[b].state = m->pstates + b;
  CK(cudaMemcpyAsync(m->pslots, m->pslots_host.data(), sizeof(DevSeq) * (bmax + 1), cudaMemcpyHostToDevice,
                     m->stream),
     "upload tile slots");
  memcpy(m->h_tokens, ids, 4ull * n);
  CK(cudaMemcpyAsync(s.d.tokens + pos, m->h_tokens, 4ull * n, cudaMemcpyHostToDevice, m->stream), "upload prompt");
  for (int done = 0; done < n;) {
    const int t = std::min(bmax, n - done);
    if ((rc = run_prefill_tile(m, t, done + t == n))) return rc;
    done += t;
  }
  CK(cudaMemcpyAsync(m->h_tokens, s.d.tokens + pos + n, 4, cudaMemcpyDeviceToHost, m->stream), "read next token");
  if ((rc = finish(m, s))) return rc;
  s.next_pos = pos + n;
  s.logits_pos = s.next_pos;
  *next_out = m->h_tokens[0];
  return TQD_OK;
}

int32_t tqd_read_logits(tqd_model* m, int32_t seq, float* host_out) {
  int32_t rc = check_model(m, seq);
  if (rc) return rc;
  if (!host_out) {
    set_error("host_out is NULL");
    return TQD_ERR_BAD_ARG;
  }
  CK(cudaMemcpyAsync(host_out, m->seqs[seq].d.logits, 4ull * m->cfg.vocab, cudaMemcpyDeviceToHost,
                     m->stream),
     "read logits");
  CK(cudaStreamSynchronize(m->stream), "synchronize");
  return TQD_OK;
}

int32_t tqd_phase_count(tqd_model* m, int32_t* out) {
  if (!m || !out) {
    set_error("model and out must be non-NULL");
    return TQD_ERR_BAD_ARG;
  }
  const int L = m->cfg.n_layers;
  *out = m->cfg.schedule == TQD_SCHED_GRAPH ? 5 * L + 2 : 4 * L + 1;
  return TQD_OK;
}

int32_t tqd_step_bytes(tqd_model* m, int32_t pos, int64_t* bytes_out) {
  if (!m || !bytes_out || pos < 0) {
    set_error("model, bytes_out and pos >= 0 required");
    return TQD_ERR_BAD_ARG;
  }
  const int64_t kv_row = (m->dm.kv16 ? 2ll : 4ll) * m->dm.kvw * 2 * m->cfg.n_layers;  // K and V, all layers
  *bytes_out = m->weight_bytes + static_cast<int64_t>(row_bytes(m->cfg.weight_type, m->cfg.hidden)) +
               kv_row * (static_cast<int64_t>(pos) + 1) + kv_row;
  return TQD_OK;
}

// ---------------------------------------------------------------- synthetic models
// The seeded generator of the synthetic inputs (synth/tqd_synth.c, linked
// into the library): input construction only, the same bytes the tests and
// the benchmark build in Python.
uint64_t tqs_stream(uint64_t seed, uint64_t tensor);
void tqs_normal_f32(uint64_t seed, uint64_t tensor, int64_t n, double mean, double sigma, float* out);
int tqs_q8_0_matrix(uint64_t seed, uint64_t tensor, int64_t rows, int64_t cols, double sigma, uint8_t* out);
int tqs_bf16_matrix(uint64_t seed, uint64_t tensor, int64_t rows, int64_t cols, double sigma, uint16_t* out);

int32_t tqd_create_synthetic(const tqd_config* cfg, uint64_t seed, void* stream, tqd_model** out) {
  if (!cfg || !out) {
    set_error("cfg and out must be non-NULL");
    return TQD_ERR_BAD_ARG;
  }
  *out = nullptr;
  if (int32_t rc = validate_config(cfg)) return rc;
  const int L = cfg->n_layers, H = cfg->hidden, hd = cfg->head_dim, I = cfg->intermediate, V = cfg->vocab;
  const int qw = cfg->n_heads * hd, kvw = cfg->n_kv_heads * hd, wt = cfg->weight_type;
  // tensor streams: the lm_head (tied embedding) 0, then per layer in this
  // order, then the final norm
  enum { kAttnNorm, kWq, kWk, kWv, kWo, kQNorm, kKNorm, kFfnNorm, kGate, kUp, kDown, kPerLayer };
  auto tensor = [&](int l, int which) { return static_cast<uint64_t>(1 + kPerLayer * l + which); };
  std::vector<std::vector<uint8_t>> mats;
  std::vector<std::vector<float>> gains;
  mats.reserve(7 * L + 1);
  gains.reserve(4 * L + 1);
  auto matrix = [&](uint64_t t, int rows, int cols) -> const void* {
    mats.emplace_back(host_row_bytes(wt, cols) * rows);
    uint8_t* p = mats.back().data();
    const int rc = wt == TQD_WEIGHT_Q8_0 ? tqs_q8_0_matrix(seed, t, rows, cols, 0.02, p)
                                         : tqs_bf16_matrix(seed, t, rows, cols, 0.02, reinterpret_cast<uint16_t*>(p));
    return rc == 0 ? p : nullptr;
  };
  auto gain = [&](uint64_t t, int n) -> const float* {
    gains.emplace_back(n);
    tqs_normal_f32(seed, t, n, 1.0, 0.1, gains.back().data());
    return gains.back().data();
  };
  std::vector<tqd_layer_weights> lw(L);
  bool ok = true;
  const void* lm = matrix(0, V, H);
  ok = ok && lm;
  for (int l = 0; l < L && ok; ++l) {
    tqd_layer_weights& w = lw[l];
    w.attn_norm = gain(tensor(l, kAttnNorm), H);
    w.wq = matrix(tensor(l, kWq), qw, H);
    w.wk = matrix(tensor(l, kWk), kvw, H);
    w.wv = matrix(tensor(l, kWv), kvw, H);
    w.wo = matrix(tensor(l, kWo), H, qw);
    w.q_norm = cfg->qk_norm ? gain(tensor(l, kQNorm), hd) : nullptr;
    w.k_norm = cfg->qk_norm ? gain(tensor(l, kKNorm), hd) : nullptr;
    w.ffn_norm = gain(tensor(l, kFfnNorm), H);
    w.w_gate = matrix(tensor(l, kGate), I, H);
    w.w_up = matrix(tensor(l, kUp), I, H);
    w.w_down = matrix(tensor(l, kDown), H, I);
    ok = w.wq && w.wk && w.wv && w.wo && w.w_gate && w.w_up && w.w_down;
  }
  if (!ok) {
    set_error("the synthetic generator refused a shape (Q8_0 needs columns %% 32 == 0)");
    return TQD_ERR_BAD_ARG;
  }
  tqd_host_weights hw{};
  hw.layers = lw.data();
  hw.out_norm = gain(static_cast<uint64_t>(1 + kPerLayer * L), H);
  hw.lm_head = lm;
  hw.embed = nullptr;  // tied
  return tqd_create(cfg, &hw, stream, out);
}

int32_t tqd_export_weights(tqd_model* m, const tqd_host_weights* out) {
  if (!m || !out || !out->layers || !out->out_norm || !out->lm_head) {
    set_error("model, out, out->layers, out->out_norm and out->lm_head must be non-NULL");
    return TQD_ERR_BAD_ARG;
  }
  if (m->poisoned) {
    set_error("model is poisoned by an earlier device error");
    return TQD_ERR_POISONED;
  }
  const tqd_config& c = m->cfg;
  const int L = c.n_layers, H = c.hidden, hd = c.head_dim, I = c.intermediate, V = c.vocab;
  const int qw = c.n_heads * hd, kvw = c.n_kv_heads * hd, wt = c.weight_type;
  for (int l = 0; l < L; ++l) {
    const tqd_layer_weights& w = out->layers[l];
    if (!w.attn_norm || !w.wq || !w.wk || !w.wv || !w.wo || !w.ffn_norm || !w.w_gate || !w.w_up || !w.w_down ||
        (c.qk_norm && (!w.q_norm || !w.k_norm))) {
      set_error("layer %d: every destination pointer must be non-NULL (q_norm, k_norm only with qk_norm)", l);
      return TQD_ERR_BAD_ARG;
    }
  }
  std::vector<uint8_t> buf;
  // `rows` device rows of `cols` columns starting at row r0, every `step`-th
  // row, into host rows in the upload format
  auto get = [&](const uint8_t* dev, int r0, int step, int rows, int cols, void* dst) -> cudaError_t {
    const size_t rb = row_bytes(wt, cols), hrb = host_row_bytes(wt, cols);
    buf.resize(rb * rows);
    cudaError_t e = cudaMemcpy2DAsync(buf.data(), rb, dev + rb * r0, rb * step, rb, rows, cudaMemcpyDeviceToHost,
                                      m->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
    if (e != cudaSuccess) return e;
    uint8_t* o = static_cast<uint8_t*>(dst);
    for (int r = 0; r < rows; ++r) {
      const uint8_t* src = buf.data() + rb * r;
      uint8_t* d = o + hrb * r;
      if (wt == TQD_WEIGHT_Q8_0) {
        for (int b = 0; b < cols / 32; ++b) {  // row layout: quants, then the blocks' f16 scales
          d[34 * b] = src[cols + 2 * b];
          d[34 * b + 1] = src[cols + 2 * b + 1];
          memcpy(d + 34 * b + 2, src + 32 * b, 32);
        }
      } else {
        memcpy(d, src, hrb);
      }
    }
    return cudaSuccess;
  };
  auto getf = [&](const float* dev, int n, const float* dst) -> cudaError_t {
    cudaError_t e = cudaMemcpyAsync(const_cast<float*>(dst), dev, 4ull * n, cudaMemcpyDeviceToHost, m->stream);
    return e == cudaSuccess ? cudaStreamSynchronize(m->stream) : e;
  };
  cudaError_t e = cudaSuccess;
  for (int l = 0; l < L && e == cudaSuccess; ++l) {
    const DevLayer& d = m->host_layers[l];
    const tqd_layer_weights& w = out->layers[l];
    void* wq = const_cast<void*>(w.wq);
    if ((e = get(d.wqkv, 0, 1, qw, H, wq)) != cudaSuccess ||
        (e = get(d.wqkv, qw, 1, kvw, H, const_cast<void*>(w.wk))) != cudaSuccess ||
        (e = get(d.wqkv, qw + kvw, 1, kvw, H, const_cast<void*>(w.wv))) != cudaSuccess ||
        (e = get(d.wo, 0, 1, H, qw, const_cast<void*>(w.wo))) != cudaSuccess ||
        (e = get(d.wgu, 0, 2, I, H, const_cast<void*>(w.w_gate))) != cudaSuccess ||
        (e = get(d.wgu, 1, 2, I, H, const_cast<void*>(w.w_up))) != cudaSuccess ||
        (e = get(d.wd, 0, 1, H, I, const_cast<void*>(w.w_down))) != cudaSuccess ||
        (e = getf(d.attn_norm, H, w.attn_norm)) != cudaSuccess || (e = getf(d.ffn_norm, H, w.ffn_norm)) != cudaSuccess)
      break;
    if (c.qk_norm && ((e = getf(d.q_norm, hd, w.q_norm)) != cudaSuccess || (e = getf(d.k_norm, hd, w.k_norm)) != cudaSuccess))
      break;
  }
  if (e == cudaSuccess) e = get(m->dm.lm_head, 0, 1, V, H, const_cast<void*>(out->lm_head));
  if (e == cudaSuccess && out->embed && m->dm.embed != m->dm.lm_head)
    e = get(m->dm.embed, 0, 1, V, H, const_cast<void*>(out->embed));
  if (e == cudaSuccess) e = getf(m->dm.out_norm, H, out->out_norm);
  if (e != cudaSuccess) return fail_cuda(m, e, "export weights");
  return TQD_OK;
}

}  // extern "C"
