// Kernels of the decode step and their launchers.
//
//  - graph schedule: one kernel per fused phase (embed; norm + QKV matvec;
//    QK-norm + RoPE + KV append + split-K attention; O matvec + residual;
//    norm + gate/up matvec + SwiGLU; down matvec + residual; norm + lm_head
//    matvec + argmax), chained with programmatic dependent launch;
//  - set-up kernels (Q8_0 repack, RoPE table) and the operator kernels.
//
// The op order is the per-layer sequence of the inferno.rs blog, "IV.4: One
// command buffer per token", section "One command buffer".
#include <climits>

#include "tqd_internal.h"
#include "tqd_phases.cuh"

namespace tqd {

// ---------------------------------------------------------------------------
// matvec: one kernel per (format, chunks per lane), chosen on the host
// ---------------------------------------------------------------------------
// The end of a full step, run by one thread of the last lm_head block: the
// argmax becomes the input token of the next position and the position
// advances ("One command buffer": the four bytes read back).
__device__ __forceinline__ void finish_step(const DevSeq& s, uint32_t pos, int winner,
                                            int max_seq) {
  int next = winner;
  if (winner == INT_MAX) {  // no candidate: every logit was NaN
    atomicOr(&s.state->err, kErrAllNaN);
    next = -1;
  }
  if (pos + 1 <= static_cast<uint32_t>(max_seq)) s.tokens[pos + 1] = next;
  s.state->last = next;
  s.state->pos = pos + 1;
  s.state->steps += 1;
}

struct MatvecKArgs {
  MatvecLaunch a;
  int cpl;
  uint32_t* err;
};

template <int FMT, int CPL>
__global__ void __launch_bounds__(kMatvecThreads) k_matvec(MatvecKArgs args) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const MatvecLaunch& a = args.a;
  float* xs = reinterpret_cast<float*>(smem_raw);
  float* red = xs + ((a.K + 3) & ~3);
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + 64);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  uint32_t parity = 0;
  if (!stage_vector(xs, a.src, a.K, bar, parity, args.err)) return;
  if (a.norm_g) rmsnorm_smem(xs, a.norm_g, a.K, a.eps, red);
  ArgmaxAcc am{-INFINITY, INT_MAX};
  const MatvecJob job{a.W, a.row_bytes, a.K, a.rows, a.epi, a.y};
  matvec_phase<FMT, CPL>(job, xs, blockIdx.x, gridDim.x, am);
  if (a.lm_head) {
    float wv;
    int wi;
    if (argmax_blocks(am, blockIdx.x, gridDim.x, a.seq.amax_v, a.seq.amax_i, a.seq.amax_count,
                      red, &wv, &wi)) {
      if (threadIdx.x == 0) finish_step(a.seq, a.seq.state->pos, wi, a.max_seq);
    }
  }
}

static cudaError_t launch_ex(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             bool pdl, bool coop, void** params) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (coop) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelExC(&cfg, fn, params);
}

cudaError_t launch_matvec(int fmt, const MatvecLaunch& a, int blocks, cudaStream_t st, bool pdl) {
  MatvecKArgs args{a, matvec_cpl(fmt, a.K), a.seq.state ? &a.seq.state->err : nullptr};
  if (args.cpl == 0 || blocks <= 0) return cudaErrorInvalidValue;
  if (a.lm_head && blocks > kMaxArgmaxBlocks) return cudaErrorInvalidValue;
  void* params[] = {&args};
  const void* fn = nullptr;
#define TQD_MV(F, C) \
  if (fmt == F && args.cpl == C) fn = reinterpret_cast<const void*>(&k_matvec<F, C>);
  TQD_MV(kFmtQ8, 1) TQD_MV(kFmtQ8, 2) TQD_MV(kFmtQ8, 4) TQD_MV(kFmtQ8, 6) TQD_MV(kFmtQ8, 8)
  TQD_MV(kFmtQ8, 12) TQD_MV(kFmtBF16, 1) TQD_MV(kFmtBF16, 2) TQD_MV(kFmtBF16, 4)
  TQD_MV(kFmtBF16, 6) TQD_MV(kFmtBF16, 8) TQD_MV(kFmtBF16, 12)
#undef TQD_MV
  if (!fn) return cudaErrorInvalidValue;
  return launch_ex(fn, dim3(blocks), dim3(kMatvecThreads), matvec_smem_bytes(a.K), st, pdl, false,
                   params);
}

// ---------------------------------------------------------------------------
// embedding: x = row `token` of the (tied) embedding, dequantised
// ("The decoder: kernels and helpers", embed_row, done on the device so the
// token never needs a host write between chained steps)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void embed_row(const DevModel& m, int tok, float* dst) {
  if (m.wtype == kFmtQ8) {
    const uint8_t* row = m.embed + static_cast<size_t>(tok) * m.row_bytes_h;
    const __half* sc = reinterpret_cast<const __half*>(row + m.H);
    for (int i = threadIdx.x; i < m.H; i += blockDim.x)
      dst[i] = __half2float(sc[i >> 5]) * static_cast<float>(static_cast<int8_t>(row[i]));
  } else {
    const uint16_t* row = reinterpret_cast<const uint16_t*>(m.embed + static_cast<size_t>(tok) * m.row_bytes_h);
    for (int i = threadIdx.x; i < m.H; i += blockDim.x)
      dst[i] = __uint_as_float(static_cast<uint32_t>(row[i]) << 16);
  }
}

__device__ __forceinline__ int checked_token(const DevModel& m, const DevSeq& s, uint32_t pos) {
  int tok = __ldcg(s.tokens + pos);
  if (tok < 0 || tok >= m.V) {
    if (threadIdx.x == 0) atomicOr(&s.state->err, kErrBadToken);
    tok = 0;
  }
  return tok;
}

__global__ void __launch_bounds__(256) k_embed(DevModel m, DevSeq s) {
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t pos = s.state->pos;
  if (pos >= static_cast<uint32_t>(m.max_seq)) {
    if (threadIdx.x == 0) atomicOr(&s.state->err, kErrCapacity);
    return;
  }
  embed_row(m, checked_token(m, s, pos), s.x);
}

cudaError_t launch_embed(const DevModel& m, const DevSeq& s, cudaStream_t st, bool pdl) {
  void* params[] = {const_cast<DevModel*>(&m), const_cast<DevSeq*>(&s)};
  return launch_ex(reinterpret_cast<const void*>(&k_embed), dim3(1), dim3(256), 0, st, pdl, false,
                   params);
}

__global__ void k_advance(DevSeq s) {
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    s.state->pos += 1;
    s.state->steps += 1;
  }
}

cudaError_t launch_advance(const DevSeq& s, cudaStream_t st, bool pdl) {
  void* params[] = {const_cast<DevSeq*>(&s)};
  return launch_ex(reinterpret_cast<const void*>(&k_advance), dim3(1), dim3(32), 0, st, pdl, false,
                   params);
}

// ---------------------------------------------------------------------------
// attention phase
// ---------------------------------------------------------------------------
__device__ __forceinline__ AttnJob layer_attn_job(const DevModel& m, const DevSeq& s, int layer,
                                                  uint32_t pos) {
  AttnJob a;
  a.q = s.qkv;
  a.k_new = s.qkv + m.qw;
  a.v_new = s.qkv + m.qw + m.kvw;
  a.q_norm = m.qk_norm ? m.layers[layer].q_norm : nullptr;
  a.k_norm = m.qk_norm ? m.layers[layer].k_norm : nullptr;
  a.rope = m.rope + static_cast<size_t>(pos) * (m.hd / 2);
  // head-major cache: [layer][kv head][position][head_dim]
  a.kc = s.kcache + static_cast<size_t>(layer) * m.max_seq * m.kvw;
  a.vc = s.vcache + static_cast<size_t>(layer) * m.max_seq * m.kvw;
  a.head_stride = static_cast<size_t>(m.max_seq) * m.hd;
  a.row_stride = static_cast<size_t>(m.hd);
  a.kv16 = m.kv16;
  if (m.kv16) {  // element offsets of an f16 cache: the layer starts half as many bytes in
    a.kc = reinterpret_cast<float*>(reinterpret_cast<__half*>(s.kcache) + static_cast<size_t>(layer) * m.max_seq * m.kvw);
    a.vc = reinterpret_cast<float*>(reinterpret_cast<__half*>(s.vcache) + static_cast<size_t>(layer) * m.max_seq * m.kvw);
  }
  a.S = static_cast<int>(pos) + 1;
  a.nq = m.nq;
  a.nkv = m.nkv;
  a.n_chunks = m.n_chunks;
  a.eps = m.eps;
  a.scale = m.attn_scale;
  a.part_o = s.part_o;
  a.part_ml = s.part_ml;
  a.count = s.attn_count;
  a.out = s.attn;
  return a;
}

// Run item `item` (kv group, chunk) of an attention job.
__device__ __forceinline__ void attention_dispatch(const AttnJob& a, int hd, int G, int item,
                                                   float* smem, uint32_t* err) {
  const int g = item / a.n_chunks, c = item - g * a.n_chunks;
  if (hd == 128) {
    switch (G) {
      case 1: attention_item<128, 1>(a, g, c, smem, err); break;
      case 2: attention_item<128, 2>(a, g, c, smem, err); break;
      case 3: attention_item<128, 3>(a, g, c, smem, err); break;
      case 4: attention_item<128, 4>(a, g, c, smem, err); break;
      default: attention_item<128, 8>(a, g, c, smem, err); break;
    }
  } else {
    switch (G) {
      case 1: attention_item<64, 1>(a, g, c, smem, err); break;
      case 2: attention_item<64, 2>(a, g, c, smem, err); break;
      case 3: attention_item<64, 3>(a, g, c, smem, err); break;
      case 4: attention_item<64, 4>(a, g, c, smem, err); break;
      default: attention_item<64, 8>(a, g, c, smem, err); break;
    }
  }
}

bool attention_supported(int hd, int group) {
  return (hd == 64 || hd == 128) &&
         (group == 1 || group == 2 || group == 3 || group == 4 || group == 8);
}

static size_t attn_smem_bytes(int hd, int G, int nwarps) {
  return static_cast<size_t>(attn_smem_floats(hd, G, nwarps)) * 4;
}

__global__ void __launch_bounds__(kAttnThreads) k_attention(DevModel m, DevSeq s, int layer) {
  extern __shared__ __align__(16) float smem_f[];
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t pos = s.state->pos;
  if (pos >= static_cast<uint32_t>(m.max_seq)) return;
  const AttnJob a = layer_attn_job(m, s, layer, pos);
  attention_dispatch(a, m.hd, m.nq / m.nkv, blockIdx.x, smem_f, &s.state->err);
}

cudaError_t launch_attention(const DevModel& m, const DevSeq& s, int layer, cudaStream_t st,
                             bool pdl) {
  void* params[] = {const_cast<DevModel*>(&m), const_cast<DevSeq*>(&s), &layer};
  const int G = m.nq / m.nkv;
  return launch_ex(reinterpret_cast<const void*>(&k_attention), dim3(m.nkv * m.n_chunks),
                   dim3(kAttnThreads), attn_smem_bytes(m.hd, G, kAttnThreads / 32), st, pdl,
                   false, params);
}

// ---------------------------------------------------------------------------
// set-up kernels
// ---------------------------------------------------------------------------
// One thread per 34-byte block: quants to the row's quant run, the scale to
// the row's scale run.  Destination row of source row r: dst_row0 + r * step.
__global__ void k_q8_repack(const uint8_t* __restrict__ src, int64_t rows, int64_t cols,
                            uint8_t* __restrict__ dst, int64_t dst_row0, int64_t dst_row_step) {
  const int64_t bpr = cols / 32;
  const int64_t nblk = rows * bpr;
  const int64_t row_bytes = static_cast<int64_t>(q8_row_bytes(cols));
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nblk;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / bpr, b = i - r * bpr;
    const uint8_t* s = src + i * 34;
    uint8_t* d = dst + (dst_row0 + r * dst_row_step) * row_bytes;
    d[cols + 2 * b] = s[0];
    d[cols + 2 * b + 1] = s[1];
#pragma unroll
    for (int j = 0; j < 32; ++j) d[32 * b + j] = s[2 + j];
  }
}

cudaError_t launch_q8_repack(const uint8_t* src_blocks, int64_t rows, int64_t cols, uint8_t* dst,
                             int64_t dst_row0, int64_t dst_row_step, cudaStream_t st) {
  const int64_t nblk = rows * (cols / 32);
  int blocks = static_cast<int>((nblk + 255) / 256);
  if (blocks > 65535) blocks = 65535;
  if (blocks < 1) blocks = 1;
  k_q8_repack<<<blocks, 256, 0, st>>>(src_blocks, rows, cols, dst, dst_row0, dst_row_step);
  return cudaGetLastError();
}

// (cos a, sin a) with a = p * theta^(-i/half), evaluated in double precision.
__global__ void k_rope_table(double theta, int half, int max_pos, float2* table) {
  const int64_t n = static_cast<int64_t>(max_pos) * half;
  for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < n;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p = k / half;
    const int i = static_cast<int>(k - p * half);
    const double a = static_cast<double>(p) * pow(theta, -static_cast<double>(i) / half);
    table[k] = make_float2(static_cast<float>(cos(a)), static_cast<float>(sin(a)));
  }
}

cudaError_t launch_rope_table(double theta, int head_dim, int max_pos, float2* table,
                              cudaStream_t st) {
  const int half = head_dim / 2;
  const int64_t n = static_cast<int64_t>(max_pos) * half;
  int blocks = static_cast<int>((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  k_rope_table<<<blocks, 256, 0, st>>>(theta, half, max_pos, table);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// operator kernels (one phase at a time, on caller memory)
// ---------------------------------------------------------------------------
cudaError_t launch_op_matvec(int fmt, const uint8_t* W, size_t row_bytes, int rows, int K,
                             const float* x, float* y, cudaStream_t st) {
  MatvecLaunch a{};
  a.W = W;
  a.row_bytes = row_bytes;
  a.K = K;
  a.rows = rows;
  a.epi = kEpiStore;
  a.y = y;
  a.src = x;
  a.norm_g = nullptr;
  a.lm_head = false;
  const int cpl = matvec_cpl(fmt, K);
  if (cpl == 0) return cudaErrorInvalidValue;
  const int R = cpl >= 4 ? 2 : 8 / cpl;
  const int groups = (rows + R - 1) / R;
  int blocks = (groups + kMatvecThreads / 32 - 1) / (kMatvecThreads / 32);
  if (blocks > 1216) blocks = 1216;
  return launch_matvec(fmt, a, blocks, st, false);
}

__global__ void __launch_bounds__(256) k_op_rmsnorm(const float* x, const float* g, int n,
                                                     float eps, float* out) {
  extern __shared__ __align__(16) float sm[];
  float* xs = sm;
  float* red = sm + ((n + 3) & ~3);
  const float* xr = x + static_cast<size_t>(blockIdx.x) * n;
  for (int i = threadIdx.x; i < n; i += blockDim.x) xs[i] = xr[i];
  __syncthreads();
  rmsnorm_smem(xs, g, n, eps, red);
  for (int i = threadIdx.x; i < n; i += blockDim.x) out[static_cast<size_t>(blockIdx.x) * n + i] = xs[i];
}

cudaError_t launch_op_rmsnorm(const float* x, const float* g, int rows, int n, float eps,
                              float* out, cudaStream_t st) {
  const size_t smem = static_cast<size_t>((n + 3) & ~3) * 4 + 64 * 4;
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  k_op_rmsnorm<<<rows, 256, smem, st>>>(x, g, n, eps, out);
  return cudaGetLastError();
}

template <int HD>
__global__ void k_op_rope(float* x, const float2* row) {
  const int lane = threadIdx.x & 31;
  float* xh = x + static_cast<size_t>(blockIdx.x) * HD;
  float v[HD / 32];
#pragma unroll
  for (int j = 0; j < HD / 32; ++j) v[j] = xh[lane + 32 * j];
  head_norm_rope<HD>(v, nullptr, row, 0.f);
#pragma unroll
  for (int j = 0; j < HD / 32; ++j) xh[lane + 32 * j] = v[j];
}

cudaError_t launch_op_rope(float* x, int n_heads, int head_dim, const float2* row,
                           cudaStream_t st) {
  if (head_dim == 128)
    k_op_rope<128><<<n_heads, 32, 0, st>>>(x, row);
  else if (head_dim == 64)
    k_op_rope<64><<<n_heads, 32, 0, st>>>(x, row);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

__global__ void __launch_bounds__(kAttnThreads) k_op_attention(AttnJob a, int hd, int G) {
  extern __shared__ __align__(16) float smem_f[];
  attention_dispatch(a, hd, G, blockIdx.x, smem_f, nullptr);
}

cudaError_t launch_op_attention(const float* q, const float* K, const float* V, int S, int nq,
                                int nkv, int hd, int n_chunks, float* out, float* part_o,
                                float* part_ml, uint32_t* count, cudaStream_t st) {
  const int G = nq / nkv;
  if (!attention_supported(hd, G)) return cudaErrorInvalidValue;
  AttnJob a{};
  a.q = q;
  a.k_new = nullptr;
  a.v_new = nullptr;
  a.q_norm = nullptr;
  a.k_norm = nullptr;
  a.rope = nullptr;
  a.kc = const_cast<float*>(K);
  a.vc = const_cast<float*>(V);
  a.head_stride = static_cast<size_t>(hd);  // K, V given as [S][n_kv * hd]
  a.row_stride = static_cast<size_t>(nkv) * hd;
  a.S = S;
  a.nq = nq;
  a.nkv = nkv;
  a.n_chunks = n_chunks;
  a.eps = 0.f;
  a.scale = static_cast<float>(1.0 / sqrt(static_cast<double>(hd)));
  a.part_o = part_o;
  a.part_ml = part_ml;
  a.count = count;
  a.out = out;
  k_op_attention<<<nkv * n_chunks, kAttnThreads, attn_smem_bytes(hd, G, kAttnThreads / 32), st>>>(
      a, hd, G);
  return cudaGetLastError();
}

__global__ void k_op_silu_mul(const float* g, const float* u, int64_t n, float* out) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = silu_mul(g[i], u[i]);
}

cudaError_t launch_op_silu_mul(const float* g, const float* u, int64_t n, float* out,
                               cudaStream_t st) {
  int blocks = static_cast<int>((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  k_op_silu_mul<<<blocks, 256, 0, st>>>(g, u, n, out);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(256) k_op_argmax(const float* x, int64_t n, int32_t* out,
                                                    float* cand_v, int32_t* cand_i,
                                                    uint32_t* count) {
  __shared__ float red[64];
  ArgmaxAcc am{-INFINITY, INT_MAX};
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    argmax_merge(am.v, am.i, x[i], static_cast<int>(i));
  warp_argmax(am.v, am.i);
  float wv;
  int wi;
  if (argmax_blocks(am, blockIdx.x, gridDim.x, cand_v, cand_i, count, red, &wv, &wi)) {
    if (threadIdx.x == 0) *out = wi == INT_MAX ? -1 : wi;
  }
}

cudaError_t launch_op_argmax(const float* x, int64_t n, int32_t* out, float* cand_v,
                             int32_t* cand_i, uint32_t* count, cudaStream_t st) {
  k_op_argmax<<<kOpArgmaxBlocks, 256, 0, st>>>(x, n, out, cand_v, cand_i, count);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- wait self-test
// Failure detection without a GPU fault: warp 0 waits on an mbarrier no thread
// arrives at (the bounded wait the ring and tensor-core kernels use); thread 32
// polls a counter nothing increments, the way a grid barrier does.  Both give
// up after kWaitLimitNs, set their error bits and return, and the context
// stays usable.
__device__ uint32_t g_wait_err;
__device__ unsigned long long g_wait_ctr;  // never incremented

__global__ void k_wait_selftest() {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    g_wait_err = 0u;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    mbar_wait_bounded(&bar, 0u, &g_wait_err);
  } else if (threadIdx.x == 32) {
    const uint64_t t0 = global_timer_ns();
    for (;;) {
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(&g_wait_ctr) : "memory");
      if (v >= 1ull) break;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicOr(&g_wait_err, kErrGridBarrier);
        break;
      }
    }
  }
}

cudaError_t run_wait_selftest(uint32_t* err_bits, cudaStream_t st) {
  k_wait_selftest<<<1, 64, 0, st>>>();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbolAsync(err_bits, g_wait_err, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(st);
}

}  // namespace tqd
