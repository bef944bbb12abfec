// Batched decode step: up to 16 sequences advance one token together, so
// every projection is a dense [rows x K] x [K x n] contraction that runs on the
// fifth-generation tensor cores (tcgen05, accumulator in tensor memory), and
// attention runs per sequence as a streaming split-K flash decode.
//
// Numerics: a Q8_0 weight w = scale * quant is exact in f32 (8-bit quant times
// an 11-bit significand), and splits exactly into two tf32 values w_hi + w_lo;
// an activation x splits into x_hi + x_lo (22 significant bits).  Three tf32
// products w_hi x_hi + w_hi x_lo + w_lo x_hi, each exact in f32 and summed in
// f32, give f32-level dot products (the dropped w_lo x_lo term is ~2^-22 of
// the product).  bf16 weights are exact in tf32, so two products suffice.
//
// What is computed is the decode step of the inferno.rs blog, "IV.4: One
// command buffer per token", for several sequences sharing one sweep of the
// weights ("Metal LLM decode", the batched prefill+decode arm).
#include <climits>

#include "tqd_internal.h"
#include "tqd_phases.cuh"

namespace tqd {
namespace {

// ---------------------------------------------------------------- tcgen05
constexpr int kTcM = 128;   // weight rows per tile (MMA M)
constexpr int kTcN = 16;    // batch columns (MMA N)
constexpr int kTcKC = 64;   // K elements per pipeline chunk
constexpr uint32_t kTileABytes = kTcM * kTcKC * 4;   // one tf32 operand chunk of A
constexpr uint32_t kTileBBytes = kTcN * kTcKC * 4;   // one tf32 operand chunk of B
constexpr uint32_t kBufBytes = 2 * kTileABytes + 2 * kTileBBytes;  // hi and lo of A and B

// Shared-memory matrix descriptor, K-major without swizzle: core matrices of
// 8 rows x 16 bytes; lbo = byte step between core matrices along K, sbo =
// byte step between 8-row groups; descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(const void* p, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((smem_addr(p) & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  return d;
}

// Instruction descriptor of kind::tf32: f32 accumulator, tf32 A and B, both
// K-major, shape M x N.
constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t dt, uint64_t ad, uint64_t bd, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(dt),
      "l"(ad), "l"(bd), "r"(idesc_tf32(kTcM, kTcN)), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// The tf32 value of an f32 (low 13 mantissa bits cleared) and the remainder.
__device__ __forceinline__ void split_tf32(float v, float& hi, float& lo) {
  hi = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
  lo = v - hi;
}

// Byte offset of element (row, k) of a chunk in the core-matrix layout with
// 16 core matrices along K (kTcKC / 4).
__device__ __forceinline__ uint32_t core_off(int row, int k) {
  return static_cast<uint32_t>(((row >> 3) * (kTcKC / 4) + (k >> 2)) * 128 + (row & 7) * 16 + (k & 3) * 4);
}

struct TcArgs {
  const uint8_t* W;     // weight rows (Q8_0 row layout, or bf16)
  size_t rb;            // bytes per weight row
  int K, rows, fmt;
  const float* X;       // activations [n][K] (row stride ldx)
  int ldx, n;
  const float* gain;    // RMSNorm gain [K] folded into the product, or nullptr
  float eps;
  int epi;              // kEpiStore / kEpiResid / kEpiSwiGLU / kEpiArgmax
  float* Y;             // outputs [n][ldy]; kEpiSwiGLU writes Y[b][row/2]
  int ldy;
  const DevSeq* seqs;   // kEpiArgmax: per-sequence logits, candidates, state
  uint32_t* count;      // kEpiArgmax: arrivals of all blocks
  uint32_t* err;
  int max_seq;
};

// One block per 128-row tile; 4 warps.  Thread t owns weight row tile*128+t
// for the dequantisation and tensor-memory lane t for the epilogue.
__global__ void __launch_bounds__(128, 1) k_tc_matmul(TcArgs a) {
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_base;
  __shared__ float inv_rms[kTcN];
  __shared__ float red_v[4][kTcN];
  __shared__ int red_i[4][kTcN];
  __shared__ uint32_t s_last;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int row = blockIdx.x * kTcM + t;
  const bool row_ok = row < a.rows;
  if (t == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;" ::"r"(
                     smem_addr(&tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // folded RMSNorm: 1/rms of every batch row (each warp four rows)
  if (a.gain) {
    for (int b = warp; b < kTcN; b += 4) {
      float ss = 0.f;
      if (b < a.n)
        for (int k = lane; k < a.K; k += 32) {
          const float v = __ldcg(a.X + static_cast<size_t>(b) * a.ldx + k);
          ss = fmaf(v, v, ss);
        }
      ss = warp_sum(ss);
      if (lane == 0) inv_rms[b] = rsqrtf(ss / static_cast<float>(a.K) + a.eps);
    }
  } else if (t < kTcN) {
    inv_rms[t] = 1.f;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t dt = tmem_base;
  const uint8_t* wrow = a.W + static_cast<size_t>(row_ok ? row : 0) * a.rb;
  const int nchunk = a.K / kTcKC;
  bool ok = true;
  uint32_t wait_parity[2] = {0u, 0u};
  for (int ci = 0; ci < nchunk; ++ci) {
    const int buf = ci & 1;
    unsigned char* base = sm + buf * kBufBytes;
    unsigned char* Ahi = base;
    unsigned char* Alo = base + kTileABytes;
    unsigned char* Bhi = base + 2 * kTileABytes;
    unsigned char* Blo = Bhi + kTileBBytes;
    if (ci >= 2) {  // the MMAs that read this buffer two chunks ago are done
      if (!mbar_wait_bounded(&bars[buf], wait_parity[buf], a.err)) ok = false;
      wait_parity[buf] ^= 1u;
    }
    const int k0 = ci * kTcKC;
    // A: this thread's row, 64 weights
    if (a.fmt == kFmtQ8) {
      const uint4* q = reinterpret_cast<const uint4*>(wrow + k0);
      const float s0 = row_ok ? __half2float(*reinterpret_cast<const __half*>(wrow + a.K + 2 * (k0 >> 5))) : 0.f;
      const float s1 = row_ok ? __half2float(*reinterpret_cast<const __half*>(wrow + a.K + 2 * ((k0 >> 5) + 1))) : 0.f;
#pragma unroll
      for (int v16 = 0; v16 < 4; ++v16) {
        const uint4 w = row_ok ? ld_weights16(q + v16) : make_uint4(0u, 0u, 0u, 0u);
        const float s = v16 < 2 ? s0 : s1;
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float f[4];
          i8x4_to_f32(words[j], f[0], f[1], f[2], f[3]);
          float4 hi, lo;
          split_tf32(f[0] * s, hi.x, lo.x);
          split_tf32(f[1] * s, hi.y, lo.y);
          split_tf32(f[2] * s, hi.z, lo.z);
          split_tf32(f[3] * s, hi.w, lo.w);
          const int k = v16 * 16 + j * 4;
          *reinterpret_cast<float4*>(Ahi + core_off(t, k)) = hi;
          *reinterpret_cast<float4*>(Alo + core_off(t, k)) = lo;
        }
      }
    } else {
      const uint4* q = reinterpret_cast<const uint4*>(wrow + 2 * k0);
#pragma unroll
      for (int v8 = 0; v8 < 8; ++v8) {
        const uint4 w = row_ok ? ld_weights16(q + v8) : make_uint4(0u, 0u, 0u, 0u);
        const int k = v8 * 8;
        *reinterpret_cast<float4*>(Ahi + core_off(t, k)) =
            make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
        *reinterpret_cast<float4*>(Ahi + core_off(t, k + 4)) =
            make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
      }
    }
    // B: 16 batch rows x 64 activations (times the norm gain), split hi / lo
    {
      const int b = t >> 3, g0 = (t & 7) * 2;
#pragma unroll
      for (int gg = 0; gg < 2; ++gg) {
        const int k = (g0 + gg) * 4;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b < a.n) x = __ldcg(reinterpret_cast<const float4*>(a.X + static_cast<size_t>(b) * a.ldx + k0 + k));
        if (a.gain) {
          const float4 g = __ldg(reinterpret_cast<const float4*>(a.gain + k0 + k));
          x.x *= g.x; x.y *= g.y; x.z *= g.z; x.w *= g.w;
        }
        float4 hi, lo;
        split_tf32(x.x, hi.x, lo.x);
        split_tf32(x.y, hi.y, lo.y);
        split_tf32(x.z, hi.z, lo.z);
        split_tf32(x.w, hi.w, lo.w);
        *reinterpret_cast<float4*>(Bhi + core_off(b, k)) = hi;
        *reinterpret_cast<float4*>(Blo + core_off(b, k)) = lo;
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (t == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      constexpr uint32_t lbo = 128, sbo = (kTcKC / 4) * 128;
#pragma unroll
      for (int s = 0; s < kTcKC / 8; ++s) {
        const uint32_t off = s * 2 * 128;
        const uint64_t ah = smem_desc(Ahi + off, lbo, sbo), al = smem_desc(Alo + off, lbo, sbo);
        const uint64_t bh = smem_desc(Bhi + off, lbo, sbo), bl = smem_desc(Blo + off, lbo, sbo);
        mma_tf32(dt, ah, bh, (ci > 0 || s > 0) ? 1u : 0u);
        mma_tf32(dt, ah, bl, 1u);
        if (a.fmt == kFmtQ8) mma_tf32(dt, al, bh, 1u);
      }
      mma_commit(&bars[buf]);
    }
  }
  // wait for the last chunk's MMAs (they complete in order)
  {
    const int last = (nchunk - 1) & 1;
    if (!mbar_wait_bounded(&bars[last], wait_parity[last], a.err)) ok = false;
  }
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  uint32_t acc[kTcN];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(acc[0]), "=r"(acc[1]), "=r"(acc[2]), "=r"(acc[3]), "=r"(acc[4]), "=r"(acc[5]),
        "=r"(acc[6]), "=r"(acc[7]), "=r"(acc[8]), "=r"(acc[9]), "=r"(acc[10]), "=r"(acc[11]),
        "=r"(acc[12]), "=r"(acc[13]), "=r"(acc[14]), "=r"(acc[15])
      : "r"(dt + (static_cast<uint32_t>(warp * 32) << 16))
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0)  // the tensor memory is released on every path
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" ::"r"(dt) : "memory");
  if (!ok) return;
  // epilogue
  float v[kTcN];
#pragma unroll
  for (int b = 0; b < kTcN; ++b) v[b] = __uint_as_float(acc[b]) * inv_rms[b];
  if (a.epi == kEpiSwiGLU) {
    // rows 2j (gate) and 2j+1 (up) sit in neighbouring lanes
#pragma unroll
    for (int b = 0; b < kTcN; ++b) {
      const float u = __shfl_down_sync(0xFFFFFFFFu, v[b], 1);
      if (b < a.n && row_ok && (row & 1) == 0) a.Y[static_cast<size_t>(b) * a.ldy + (row >> 1)] = silu_mul(v[b], u);
    }
    return;
  }
  if (a.epi != kEpiArgmax) {
    if (row_ok)
      for (int b = 0; b < a.n; ++b) {
        float* y = a.Y + static_cast<size_t>(b) * a.ldy + row;
        *y = a.epi == kEpiResid ? *y + v[b] : v[b];
      }
    return;
  }
  // lm_head: logits and the argmax of every sequence
#pragma unroll
  for (int b = 0; b < kTcN; ++b) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    if (b < a.n && row_ok) {
      a.seqs[b].logits[row] = v[b];
      bv = v[b];
      bi = row;
    }
    warp_argmax(bv, bi);
    if (lane == 0) {
      red_v[warp][b] = bv;
      red_i[warp][b] = bi;
    }
  }
  __syncthreads();
  if (t < a.n) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int w = 0; w < 4; ++w) argmax_merge(bv, bi, red_v[w][t], red_i[w][t]);
    a.seqs[t].amax_v[blockIdx.x] = bv;
    a.seqs[t].amax_i[blockIdx.x] = bi;
  }
  __syncthreads();
  if (t == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(a.count, 1u);
    s_last = old == gridDim.x - 1u;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  // one warp per sequence reduces the blocks' candidates
  for (int b = warp; b < a.n; b += 4) {
    const DevSeq& s = a.seqs[b];
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int k = lane; k < static_cast<int>(gridDim.x); k += 32)
      argmax_merge(bv, bi, __ldcg(s.amax_v + k), __ldcg(s.amax_i + k));
    warp_argmax(bv, bi);
    if (lane == 0) {
      const uint32_t pos = s.state->pos;
      int next = bi;
      if (bi == INT_MAX) {
        atomicOr(&s.state->err, kErrAllNaN);
        next = -1;
      }
      if (pos + 1 <= static_cast<uint32_t>(a.max_seq)) s.tokens[pos + 1] = next;
      s.state->pos = pos + 1;
      s.state->steps += 1;
    }
  }
  if (t == 0) *a.count = 0u;
}

// ---------------------------------------------------------------- embedding
__global__ void __launch_bounds__(256) k_embed_batch(DevModel m, const DevSeq* seqs, int n, float* X) {
  const int b = blockIdx.x;
  if (b >= n) return;
  const DevSeq& s = seqs[b];
  const uint32_t pos = s.state->pos;
  if (pos >= static_cast<uint32_t>(m.max_seq)) {
    if (threadIdx.x == 0) atomicOr(&s.state->err, kErrCapacity);
    return;
  }
  int tok = __ldcg(s.tokens + pos);
  if (tok < 0 || tok >= m.V) {
    if (threadIdx.x == 0) atomicOr(&s.state->err, kErrBadToken);
    tok = 0;
  }
  float* x = X + static_cast<size_t>(b) * m.H;
  if (m.wtype == kFmtQ8) {
    const uint8_t* row = m.embed + static_cast<size_t>(tok) * m.row_bytes_h;
    const __half* sc = reinterpret_cast<const __half*>(row + m.H);
    for (int i = threadIdx.x; i < m.H; i += blockDim.x)
      x[i] = __half2float(sc[i >> 5]) * static_cast<float>(static_cast<int8_t>(row[i]));
  } else {
    const uint16_t* row = reinterpret_cast<const uint16_t*>(m.embed + static_cast<size_t>(tok) * m.row_bytes_h);
    for (int i = threadIdx.x; i < m.H; i += blockDim.x)
      x[i] = __uint_as_float(static_cast<uint32_t>(row[i]) << 16);
  }
}

// ---------------------------------------------------------------- attention
// One block per (sequence, kv head, chunk): a producer thread streams the
// chunk's cached K/V rows into a small shared-memory ring with bulk copies;
// eight consumer warps run the online softmax; the last chunk of a (sequence,
// kv head) combines the chunks ("Eight kernels", attention_decode, as a
// split-K flash decode).
constexpr int kAW = 8;                  // consumer warps
constexpr int kAT = kAW * 32;           // consumer threads
constexpr int kASlots = 3;
constexpr uint32_t kASlotBytes = 32 * 1024;

__device__ __forceinline__ void async() { asm volatile("bar.sync 1, %0;" ::"n"(kAT) : "memory"); }

template <int HD, int G>
__device__ void attn_batch_item(const DevModel& m, const DevSeq& s, int layer, int g, int c, int nch,
                                const float* qkv, float* attn, unsigned char* sm) {
  constexpr int NJ = HD / 32, DPL = HD / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kASlots * kASlotBytes);
  uint64_t* empty = full + kASlots;
  float* qs = reinterpret_cast<float*>(empty + kASlots);  // [G][HD]
  float* knew = qs + G * HD;
  float* vnew = knew + HD;
  float* wst = vnew + HD;                                   // [kAW][G][HD + 2]
  const uint32_t pos = s.state->pos;
  const int S = static_cast<int>(pos) + 1;
  const int cs = (S + nch - 1) / nch;
  const int t0 = min(S, c * cs), t1 = min(S, t0 + cs);
  const bool has_new = t0 <= static_cast<int>(pos) && static_cast<int>(pos) < t1;
  const int tc = min(t1, static_cast<int>(pos));
  const int rpp = static_cast<int>(kASlotBytes / (2u * 4u * HD));
  const size_t head = (static_cast<size_t>(layer) * m.nkv + g) * m.max_seq * HD;
  uint32_t* err = &s.state->err;
  if (threadIdx.x == kAT) {
    // producer
    uint32_t n = 0;
    for (int a0 = t0; a0 < tc; a0 += rpp, ++n) {
      const int cnt = min(rpp, tc - a0);
      const uint32_t slot = n % kASlots, use = n / kASlots;
      if (use > 0 && !mbar_wait_bounded(empty + slot, (use - 1) & 1u, err)) break;
      const uint32_t bytes = static_cast<uint32_t>(cnt) * HD * 4u;
      unsigned char* dst = sm + slot * kASlotBytes;
      mbar_arrive_expect_tx(full + slot, 2u * bytes);
      bulk_g2s(dst, s.kcache + head + static_cast<size_t>(a0) * HD, bytes, full + slot);
      bulk_g2s(dst + static_cast<size_t>(rpp) * HD * 4u, s.vcache + head + static_cast<size_t>(a0) * HD, bytes,
               full + slot);
    }
    return;
  }
  if (threadIdx.x > kAT) return;
  const DevLayer& L = m.layers[layer];
  const float2* rope = m.rope + static_cast<size_t>(pos) * (HD / 2);
  if (warp < G) {
    const int h = g * G + warp;
    float v[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) v[j] = __ldcg(qkv + h * HD + lane + 32 * j);
    head_norm_rope<HD>(v, m.qk_norm ? L.q_norm : nullptr, rope, m.eps);
#pragma unroll
    for (int j = 0; j < NJ; ++j) qs[warp * HD + lane + 32 * j] = v[j];
  } else if (warp == kAW - 1 && has_new) {
    float kv[NJ], vv[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      kv[j] = __ldcg(qkv + m.qw + g * HD + lane + 32 * j);
      vv[j] = __ldcg(qkv + m.qw + m.kvw + g * HD + lane + 32 * j);
    }
    head_norm_rope<HD>(kv, m.qk_norm ? L.k_norm : nullptr, rope, m.eps);
    const size_t r = head + static_cast<size_t>(pos) * HD;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      s.kcache[r + lane + 32 * j] = kv[j];
      s.vcache[r + lane + 32 * j] = vv[j];
      knew[lane + 32 * j] = kv[j];
      vnew[lane + 32 * j] = vv[j];
    }
  }
  async();
  float qv[G][DPL], mm[G], ll[G], oo[G][DPL];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    mm[hh] = -INFINITY;
    ll[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      qv[hh][e] = qs[hh * HD + lane * DPL + e];
      oo[hh][e] = 0.f;
    }
  }
  auto row_update = [&](const float* kr, const float* vr) {
    float kf[DPL], vf[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      kf[e] = kr[lane * DPL + e];
      vf[e] = vr[lane * DPL + e];
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) d = fmaf(qv[hh][e], kf[e], d);
      const float sc = warp_sum(d) * m.attn_scale;
      if (sc > mm[hh]) {
        const float corr = expf(mm[hh] - sc);
        mm[hh] = sc;
        ll[hh] = ll[hh] * corr + 1.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) oo[hh][e] = fmaf(oo[hh][e], corr, vf[e]);
      } else {
        const float p = expf(sc - mm[hh]);
        ll[hh] += p;
#pragma unroll
        for (int e = 0; e < DPL; ++e) oo[hh][e] = fmaf(p, vf[e], oo[hh][e]);
      }
    }
  };
  uint32_t n = 0;
  for (int a0 = t0; a0 < tc; a0 += rpp, ++n) {
    const int cnt = min(rpp, tc - a0);
    const uint32_t slot = n % kASlots;
    mbar_wait_bounded(full + slot, (n / kASlots) & 1u, err);
    const float* Ks = reinterpret_cast<const float*>(sm + slot * kASlotBytes);
    const float* Vs = Ks + static_cast<size_t>(rpp) * HD;
    for (int r = warp; r < cnt; r += kAW) row_update(Ks + r * HD, Vs + r * HD);
    __syncwarp();
    if (lane == 0)
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(empty + slot)) : "memory");
  }
  if (has_new && warp == ((tc - t0) % kAW)) row_update(knew, vnew);
  const int stride = HD + 2;
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    float* w = wst + (warp * G + hh) * stride;
#pragma unroll
    for (int e = 0; e < DPL; ++e) w[lane * DPL + e] = oo[hh][e];
    if (lane == 0) {
      w[HD] = mm[hh];
      w[HD + 1] = ll[hh];
    }
  }
  async();
  for (int idx = threadIdx.x; idx < G * HD; idx += kAT) {
    const int hh = idx / HD, d = idx - hh * HD;
    float M = -INFINITY;
    for (int w = 0; w < kAW; ++w) M = fmaxf(M, wst[(w * G + hh) * stride + HD]);
    float O = 0.f, Ls = 0.f;
    if (M != -INFINITY)
      for (int w = 0; w < kAW; ++w) {
        const float* ws = wst + (w * G + hh) * stride;
        const float f = expf(ws[HD] - M);
        O = fmaf(f, ws[d], O);
        Ls = fmaf(f, ws[HD + 1], Ls);
      }
    const int h = g * G + hh;
    s.part_o[(static_cast<size_t>(h) * nch + c) * HD + d] = O;
    if (d == 0) {
      s.part_ml[(static_cast<size_t>(h) * nch + c) * 2] = M;
      s.part_ml[(static_cast<size_t>(h) * nch + c) * 2 + 1] = Ls;
    }
  }
  async();
  __shared__ uint32_t s_last;
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(s.attn_count + g, 1u);
    s_last = old == static_cast<uint32_t>(nch) - 1u;
    if (s_last) __threadfence();
  }
  async();
  if (!s_last) return;
  for (int idx = threadIdx.x; idx < G * HD; idx += kAT) {
    const int hh = idx / HD, d = idx - hh * HD;
    const int h = g * G + hh;
    const float* ml = s.part_ml + static_cast<size_t>(h) * nch * 2;
    const float* po = s.part_o + static_cast<size_t>(h) * nch * HD;
    float M = -INFINITY;
    for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(ml + 2 * cc));
    float num = 0.f, den = 0.f;
    for (int cc = 0; cc < nch; ++cc) {
      const float mc = __ldcg(ml + 2 * cc);
      if (mc == -INFINITY) continue;
      const float f = expf(mc - M);
      num = fmaf(f, __ldcg(po + static_cast<size_t>(cc) * HD + d), num);
      den = fmaf(f, __ldcg(ml + 2 * cc + 1), den);
    }
    attn[h * HD + d] = num / den;
  }
  async();
  if (threadIdx.x == 0) s.attn_count[g] = 0u;
}

__global__ void __launch_bounds__(kAT + 32, 1)
    k_attn_batch(DevModel m, const DevSeq* seqs, int layer, int nch, const float* QKV, float* ATTN) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const int per_seq = m.nkv * nch;
  const int b = blockIdx.x / per_seq, item = blockIdx.x - b * per_seq;
  const int g = item / nch, c = item - g * nch;
  const DevSeq& s = seqs[b];
  if (threadIdx.x == 0) {
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + kASlots * kASlotBytes);
    for (int i = 0; i < kASlots; ++i) {
      mbar_init(full + i, 1);
      mbar_init(full + kASlots + i, kAW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (s.state->pos >= static_cast<uint32_t>(m.max_seq)) return;
  const float* qkv = QKV + static_cast<size_t>(b) * (m.qw + 2 * m.kvw);
  float* attn = ATTN + static_cast<size_t>(b) * m.qw;
  const int G = m.nq / m.nkv;
  if (m.hd == 128) {
    switch (G) {
      case 1: attn_batch_item<128, 1>(m, s, layer, g, c, nch, qkv, attn, sm); break;
      case 2: attn_batch_item<128, 2>(m, s, layer, g, c, nch, qkv, attn, sm); break;
      case 3: attn_batch_item<128, 3>(m, s, layer, g, c, nch, qkv, attn, sm); break;
      default: attn_batch_item<128, 4>(m, s, layer, g, c, nch, qkv, attn, sm); break;
    }
  } else {
    switch (G) {
      case 1: attn_batch_item<64, 1>(m, s, layer, g, c, nch, qkv, attn, sm); break;
      case 2: attn_batch_item<64, 2>(m, s, layer, g, c, nch, qkv, attn, sm); break;
      case 3: attn_batch_item<64, 3>(m, s, layer, g, c, nch, qkv, attn, sm); break;
      default: attn_batch_item<64, 4>(m, s, layer, g, c, nch, qkv, attn, sm); break;
    }
  }
}

size_t attn_batch_smem(const DevModel& m) {
  const int G = m.nq / m.nkv;
  return kASlots * kASlotBytes + 16 * kASlots +
         4u * (G * m.hd + 2 * m.hd + kAW * G * (m.hd + 2));
}

size_t tc_smem() { return 2 * static_cast<size_t>(kBufBytes); }

}  // namespace

int batch_max() { return kTcN; }

bool batch_supported(const DevModel& m) {
  const int G = m.nq / m.nkv;
  return G >= 1 && G <= 4 && (m.hd == 64 || m.hd == 128) && m.H % kTcKC == 0 &&
         m.qw % kTcKC == 0 && m.I % kTcKC == 0 && attn_batch_smem(m) <= 227 * 1024;
}

cudaError_t batch_setup(const DevModel& m) {
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&k_tc_matmul),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(tc_smem()));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(&k_attn_batch),
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(attn_batch_smem(m)));
}

// One batched step for sequences seqs[0..n): embedding, every layer, lm_head
// and argmax; `full` = false skips the lm_head (then pos is advanced by the
// caller's kernel).  X, QKV, ATTN, H are batch activations.
cudaError_t enqueue_batch_step(const DevModel& m, const DevLayer* host_layers, const DevSeq* seqs,
                               int n, int nch, float* X, float* QKV, float* ATTN, float* H,
                               uint32_t* count, uint32_t* err, cudaStream_t st) {
  k_embed_batch<<<n, 256, 0, st>>>(m, seqs, n, X);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int fmt = m.wtype;
  auto mm = [&](const uint8_t* W, size_t rb, int K, int rows, const float* Xin, int ldx,
                const float* gain, int epi, float* Y, int ldy) {
    TcArgs a{};
    a.W = W; a.rb = rb; a.K = K; a.rows = rows; a.fmt = fmt;
    a.X = Xin; a.ldx = ldx; a.n = n; a.gain = gain; a.eps = m.eps;
    a.epi = epi; a.Y = Y; a.ldy = ldy; a.seqs = seqs; a.count = count; a.err = err;
    a.max_seq = m.max_seq;
    const int tiles = (rows + kTcM - 1) / kTcM;
    k_tc_matmul<<<tiles, 128, tc_smem(), st>>>(a);
    return cudaGetLastError();
  };
  const int lqkv = m.qw + 2 * m.kvw;
  for (int l = 0; l < m.n_layers; ++l) {
    const DevLayer& L = host_layers[l];
    if ((e = mm(L.wqkv, m.row_bytes_h, m.H, lqkv, X, m.H, L.attn_norm, kEpiStore, QKV, lqkv)) != cudaSuccess)
      return e;
    k_attn_batch<<<n * m.nkv * nch, kAT + 32, attn_batch_smem(m), st>>>(m, seqs, l, nch, QKV, ATTN);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = mm(L.wo, m.row_bytes_qw, m.qw, m.H, ATTN, m.qw, nullptr, kEpiResid, X, m.H)) != cudaSuccess)
      return e;
    if ((e = mm(L.wgu, m.row_bytes_h, m.H, 2 * m.I, X, m.H, L.ffn_norm, kEpiSwiGLU, H, m.I)) != cudaSuccess)
      return e;
    if ((e = mm(L.wd, m.row_bytes_i, m.I, m.H, H, m.I, nullptr, kEpiResid, X, m.H)) != cudaSuccess)
      return e;
  }
  return mm(m.lm_head, m.row_bytes_h, m.H, m.V, X, m.H, m.out_norm, kEpiArgmax, nullptr, 0);
}

}  // namespace tqd
