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
// One CTA computes a 128-row tile of W against the n <= 16 activation rows
// over a K range; the tile's K is split over the CTAs of one cluster, whose
// partial sums are reduced through distributed shared memory in a fixed order
// (deterministic).  Operands are bf16 (kind::f16, f32 accumulation):
//   A = the int8 quants, exact in bf16; every 32-wide Q8_0 block accumulates
//       into its own 16 tensor-memory columns, and its f16 scale multiplies
//       the block's column sum when the accumulator is read out (bf16
//       weights: the same layout with scale 1);
//   B = x (times the RMSNorm gain) split into three bf16 parts x1 + x2 + x3
//       (each the rounding of what the previous ones left), 24 significant
//       bits, so the products are exact and the sums are f32 sums.
constexpr int kMmThreads = 128;        // 4 warps; thread t owns weight row t of the tile
constexpr int kTcM = 128;              // weight rows per tile (MMA M)
constexpr int kTcN = 16;               // batch columns (MMA N)
constexpr int kSubK = 64;              // K elements per MMA sub-chunk
constexpr int kPassBytes = 128;        // weight bytes per row per pass (Q8_0: 128 K, bf16: 64 K)
constexpr int kRawStride = kPassBytes + 16;  // padded row: conflict-free 16-byte reads
constexpr int kRawStages = 2;
constexpr uint32_t kRawBytes = kTcM * kRawStride;
constexpr uint32_t kABytes = kTcM * kSubK * 2;       // one bf16 A sub-chunk
constexpr uint32_t kBPartBytes = kTcN * kSubK * 2;   // one bf16 part of B
constexpr uint32_t kBBytes = 3 * kBPartBytes;
constexpr int kRedStride = kTcN + 1;
constexpr uint32_t kOffA = kRawStages * kRawBytes;
constexpr uint32_t kOffB = kOffA + 2 * kABytes;
constexpr uint32_t kOffRed = kOffB + 2 * kBBytes;
constexpr uint32_t kMmSmem = kOffRed + kTcM * kRedStride * 4;
constexpr uint32_t kTmemCols = 128;    // two passes x four blocks x 16 columns
constexpr int kMaxCluster = 8;

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

// Instruction descriptor of kind::f16 with bf16 A and B, f32 accumulator,
// both K-major, shape M x N.
constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t dt, uint64_t ad, uint64_t bd, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dt),
      "l"(ad), "l"(bd), "r"(idesc_bf16(kTcM, kTcN)), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// Byte offset of element (row, k) of a bf16 sub-chunk in the core-matrix
// layout with kSubK / 8 core matrices along K.
__device__ __forceinline__ uint32_t core_off16(int row, int k) {
  return static_cast<uint32_t>(((row >> 3) * (kSubK / 8) + (k >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

// Four int8 (one word) -> four bf16 (two words), exact.
__device__ __forceinline__ void i8x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  float f0, f1, f2, f3;
  i8x4_to_f32(w, f0, f1, f2, f3);
  lo = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
  hi = __byte_perm(__float_as_uint(f2), __float_as_uint(f3), 0x7632);
}

// x = x1 + x2 + x3 + (a remainder below 2^-24 |x|), each part bf16.
__device__ __forceinline__ void split3_bf16(float x, uint32_t& p1, uint32_t& p2, uint32_t& p3) {
  const __nv_bfloat16 h1 = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(h1);
  const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(h2);
  p1 = __bfloat16_as_ushort(h1);
  p2 = __bfloat16_as_ushort(h2);
  p3 = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// A float in the shared memory of CTA `cta` of the cluster, at the offset of p.
__device__ __forceinline__ float ld_dsmem(const float* p, uint32_t cta) {
  uint32_t a;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(cta));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ void tmem_ld16(uint32_t addr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(addr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

struct MmArgs {
  const uint8_t* W;     // weight rows (Q8_0 row layout, or bf16)
  size_t rb;            // bytes per weight row
  int K, rows, fmt;
  int cs;               // CTAs per tile (the cluster), each over K / cs columns
  const float* X;       // activations [n][ldx]
  int ldx, n;
  const float* gain;    // RMSNorm gain folded into the product, or nullptr
  const float* ss;      // with gain: [nss][16] partial sums of squares of the X rows
  int nss;
  float eps;
  int epi;              // kEpiStore / kEpiResid / kEpiSwiGLU / kEpiArgmax
  float* Y;             // outputs [n][ldy]; kEpiResid adds in place; kEpiSwiGLU writes Y[b][row/2]
  int ldy;
  float* ss_out;        // kEpiResid: [gridDim.x][16] partial sums of squares of the new rows, or nullptr
  const DevSeq* seqs;   // kEpiArgmax: per-sequence logits, candidates, state
  uint32_t* count;      // kEpiArgmax: arrivals of all blocks
  uint32_t* err;
  int max_seq;
};

__global__ void __launch_bounds__(kMmThreads, 1) k_mm16(MmArgs a) {
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ __align__(8) uint64_t bars[4];  // [0..1] sub-chunk buffers free, [2..3] a pass's sums ready
  __shared__ uint32_t tmem_base;
  __shared__ float inv_rms[kTcN];
  __shared__ float wred_v[4][kTcN];
  __shared__ int wred_i[4][kTcN];
  __shared__ uint32_t s_last;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int rank = static_cast<int>(cluster_rank()), tile = blockIdx.x / a.cs;
  const int row0 = tile * kTcM, row = row0 + t;
  const bool row_ok = row < a.rows;
  const bool q8 = a.fmt == kFmtQ8;
  const int KR = a.K / a.cs, kc0 = rank * KR;
  const int PK = q8 ? kPassBytes : kPassBytes / 2;  // K per pass
  const int npass = (KR + PK - 1) / PK;
  // weight bytes of pass p for all 128 rows -> raw stage p % kRawStages
  auto issue_raw = [&](int p) {
    const int k0 = kc0 + p * PK, pk = min(PK, kc0 + KR - k0);
    const int chunks = (q8 ? pk : 2 * pk) / 16;
    unsigned char* dst = sm + (p % kRawStages) * kRawBytes;
    for (int c = t; c < kTcM * 8; c += kMmThreads) {
      const int r = c >> 3, ch = c & 7;
      if (ch < chunks) {
        const bool ok = row0 + r < a.rows;
        const uint8_t* src = a.W + static_cast<size_t>(ok ? row0 + r : 0) * a.rb + (q8 ? k0 : 2 * k0) + ch * 16;
        cp_async16(dst + r * kRawStride + ch * 16, src, ok);
      }
    }
    cp_async_commit();
  };
  if (t == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base)), "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // weights never depend on earlier kernels: their loads start before the wait
  issue_raw(0);
  if (npass > 1) issue_raw(1);
  pdl_wait();
  pdl_launch_dependents();
  if (t < kTcN) {
    float r = 1.f;
    if (a.gain) {
      float ss = 0.f;
#pragma unroll 8
      for (int i = 0; i < a.nss; ++i) ss += __ldcg(a.ss + i * kTcN + t);
      r = rsqrtf(ss / static_cast<float>(a.K) + a.eps);
    }
    inv_rms[t] = r;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t dt = tmem_base;
  const uint32_t lane_addr = dt + (static_cast<uint32_t>(warp * 32) << 16);
  float acc[kTcN];
#pragma unroll
  for (int b = 0; b < kTcN; ++b) acc[b] = 0.f;
  float s_cur[4], s_prev[4];
  uint32_t ph[4] = {0u, 0u, 0u, 0u};
  bool ok = true;
  int sub = 0, nblk_prev = 0;
  // read out pass q: scale each block's column sums and add them up
  auto readout = [&](int q, const float (&sc)[4], int nblk) {
    if (!mbar_wait_bounded(&bars[2 + (q & 1)], ph[2 + (q & 1)], a.err)) ok = false;
    ph[2 + (q & 1)] ^= 1u;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    for (int blk = 0; blk < nblk; ++blk) {
      float v[16];
      tmem_ld16(lane_addr + (q & 1) * 64 + blk * 16, v);
#pragma unroll
      for (int b = 0; b < kTcN; ++b) acc[b] = fmaf(sc[blk], v[b], acc[b]);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  };
  for (int p = 0; p < npass; ++p) {
    const int k0 = kc0 + p * PK, pk = min(PK, kc0 + KR - k0);
    const int nblk = pk / 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s_cur[i] = 1.f;
      if (q8) {
        s_cur[i] = 0.f;
        if (row_ok && i < nblk)
          s_cur[i] = __half2float(__ushort_as_half(ld_weights_u16(a.W + static_cast<size_t>(row) * a.rb + a.K +
                                                                   2 * (k0 / 32 + i))));
      }
    }
    if (p + 1 < npass) cp_async_wait<1>();
    else cp_async_wait<0>();
    __syncthreads();
    const unsigned char* raw = sm + (p % kRawStages) * kRawBytes + t * kRawStride;
    const int nsub = (pk + kSubK - 1) / kSubK;
    for (int j = 0; j < nsub; ++j, ++sub) {
      const int u = sub & 1;
      const int sk = min(kSubK, pk - j * kSubK);  // 64 or 32
      if (sub >= 2) {
        if (!mbar_wait_bounded(&bars[u], ph[u], a.err)) ok = false;
        ph[u] ^= 1u;
      }
      unsigned char* A = sm + kOffA + u * kABytes;
      unsigned char* B = sm + kOffB + u * kBBytes;
      {  // B: 16 batch rows x sk activations (times the gain), three bf16 parts
        const int b = t >> 3, k8 = (t & 7) * 8;
        if (k8 < sk) {
          const int kg = k0 + j * kSubK + k8;
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.f;
          if (b < a.n) {
            const float4 x0 = __ldcg(reinterpret_cast<const float4*>(a.X + static_cast<size_t>(b) * a.ldx + kg));
            const float4 x1 = __ldcg(reinterpret_cast<const float4*>(a.X + static_cast<size_t>(b) * a.ldx + kg + 4));
            x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
            x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
            if (a.gain) {
              const float4 g0 = __ldg(reinterpret_cast<const float4*>(a.gain + kg));
              const float4 g1 = __ldg(reinterpret_cast<const float4*>(a.gain + kg + 4));
              x[0] *= g0.x; x[1] *= g0.y; x[2] *= g0.z; x[3] *= g0.w;
              x[4] *= g1.x; x[5] *= g1.y; x[6] *= g1.z; x[7] *= g1.w;
            }
          }
          uint32_t p1[8], p2[8], p3[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) split3_bf16(x[e], p1[e], p2[e], p3[e]);
          const uint32_t off = core_off16(b, k8);
          *reinterpret_cast<uint4*>(B + off) =
              make_uint4(p1[0] | (p1[1] << 16), p1[2] | (p1[3] << 16), p1[4] | (p1[5] << 16), p1[6] | (p1[7] << 16));
          *reinterpret_cast<uint4*>(B + kBPartBytes + off) =
              make_uint4(p2[0] | (p2[1] << 16), p2[2] | (p2[3] << 16), p2[4] | (p2[5] << 16), p2[6] | (p2[7] << 16));
          *reinterpret_cast<uint4*>(B + 2 * kBPartBytes + off) =
              make_uint4(p3[0] | (p3[1] << 16), p3[2] | (p3[3] << 16), p3[4] | (p3[5] << 16), p3[6] | (p3[7] << 16));
        }
      }
      // A: this thread's row of the sub-chunk as bf16
      if (q8) {
        for (int v = 0; v < sk / 16; ++v) {
          const uint4 w = *reinterpret_cast<const uint4*>(raw + j * kSubK + v * 16);
          uint32_t o[8];
          i8x4_to_bf16x4(w.x, o[0], o[1]);
          i8x4_to_bf16x4(w.y, o[2], o[3]);
          i8x4_to_bf16x4(w.z, o[4], o[5]);
          i8x4_to_bf16x4(w.w, o[6], o[7]);
          *reinterpret_cast<uint4*>(A + core_off16(t, v * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(A + core_off16(t, v * 16 + 8)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
      } else {
        for (int v = 0; v < sk / 8; ++v)
          *reinterpret_cast<uint4*>(A + core_off16(t, v * 8)) =
              *reinterpret_cast<const uint4*>(raw + 2 * j * kSubK + v * 16);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
      if (t == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t col0 = (p & 1) * 64;
        for (int bk = 0; bk < sk / 32; ++bk) {
          const uint32_t d = dt + col0 + (j * 2 + bk) * 16;
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            const uint32_t koff = (bk * 2 + ks) * 256;  // 16 K = two core matrices
            const uint64_t ad = smem_desc(A + koff, 128, (kSubK / 8) * 128);
#pragma unroll
            for (int pt = 0; pt < 3; ++pt)
              mma_bf16(d, ad, smem_desc(B + pt * kBPartBytes + koff, 128, (kSubK / 8) * 128),
                       (ks | pt) ? 1u : 0u);
          }
        }
        mma_commit(&bars[u]);
        if (j == nsub - 1) mma_commit(&bars[2 + (p & 1)]);
      }
    }
    // every thread is past its last read of this raw stage: refill it
    if (p + kRawStages < npass) issue_raw(p + kRawStages);
    if (p > 0) readout(p - 1, s_prev, nblk_prev);
#pragma unroll
    for (int i = 0; i < 4; ++i) s_prev[i] = s_cur[i];
    nblk_prev = nblk;
  }
  readout(npass - 1, s_prev, nblk_prev);
  __syncthreads();
  if (warp == 0) {  // the tensor memory is released on every path
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(dt), "n"(kTmemCols) : "memory");
  }
  (void)ok;  // a timed-out wait has set the error word; the host reports it
  // cluster reduction of the K partials, then the epilogue; thread t handles
  // row pairs (2m, 2m+1) of this CTA's share of the tile for sequence t % 16
  float* red = reinterpret_cast<float*>(sm + kOffRed);
#pragma unroll
  for (int b = 0; b < kTcN; ++b) red[t * kRedStride + b] = acc[b];
  cluster_sync();
  const int rpc = kTcM / a.cs;
  const int b = t & (kTcN - 1);
  const float sc = inv_rms[b];
  float ssum = 0.f, bv = -INFINITY;
  int bi = INT_MAX;
  for (int idx = t; idx < rpc * (kTcN / 2); idx += kMmThreads) {
    const int lr = rank * rpc + 2 * (idx / kTcN);
    float v0 = 0.f, v1 = 0.f;
    for (int q = 0; q < a.cs; ++q) {
      v0 += ld_dsmem(red + lr * kRedStride + b, static_cast<uint32_t>(q));
      v1 += ld_dsmem(red + (lr + 1) * kRedStride + b, static_cast<uint32_t>(q));
    }
    v0 *= sc;
    v1 *= sc;
    const int r0 = row0 + lr, r1 = r0 + 1;
    if (b >= a.n || r0 >= a.rows) continue;
    const bool ok1 = r1 < a.rows;
    if (a.epi == kEpiSwiGLU) {
      a.Y[static_cast<size_t>(b) * a.ldy + (r0 >> 1)] = silu_mul(v0, v1);
    } else if (a.epi == kEpiArgmax) {
      float* lg = a.seqs[b].logits;
      lg[r0] = v0;
      argmax_merge(bv, bi, v0, r0);
      if (ok1) {
        lg[r1] = v1;
        argmax_merge(bv, bi, v1, r1);
      }
    } else {
      float* y = a.Y + static_cast<size_t>(b) * a.ldy;
      if (a.epi == kEpiResid) {
        v0 += y[r0];
        if (ok1) v1 += y[r1];
        ssum = fmaf(v0, v0, ssum);
        if (ok1) ssum = fmaf(v1, v1, ssum);
      }
      y[r0] = v0;
      if (ok1) y[r1] = v1;
    }
  }
  cluster_sync();  // the cluster's partials are no longer read
  if (a.epi == kEpiResid && a.ss_out) {
    ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, 16);
    if (lane < kTcN) wred_v[warp][lane] = ssum;
    __syncthreads();
    if (t < kTcN) a.ss_out[blockIdx.x * kTcN + t] = wred_v[0][t] + wred_v[1][t] + wred_v[2][t] + wred_v[3][t];
    return;
  }
  if (a.epi != kEpiArgmax) return;
  // lm_head: this block's candidate per sequence, then the last block to
  // arrive picks every sequence's winner
  {
    const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, 16);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, 16);
    argmax_merge(bv, bi, ov, oi);
    if (lane < kTcN) {
      wred_v[warp][lane] = bv;
      wred_i[warp][lane] = bi;
    }
  }
  __syncthreads();
  if (t < a.n) {
    float cv = -INFINITY;
    int ci = INT_MAX;
    for (int w = 0; w < 4; ++w) argmax_merge(cv, ci, wred_v[w][t], wred_i[w][t]);
    a.seqs[t].amax_v[blockIdx.x] = cv;
    a.seqs[t].amax_i[blockIdx.x] = ci;
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
  for (int q = warp; q < a.n; q += 4) {
    const DevSeq& s = a.seqs[q];
    float cv = -INFINITY;
    int ci = INT_MAX;
    for (int k = lane; k < static_cast<int>(gridDim.x); k += 32)
      argmax_merge(cv, ci, __ldcg(s.amax_v + k), __ldcg(s.amax_i + k));
    warp_argmax(cv, ci);
    if (lane == 0) {
      const uint32_t pos = s.state->pos;
      int next = ci;
      if (ci == INT_MAX) {
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

// CTAs per tile for K columns: the largest of 8, 4, 2, 1 whose share of K is
// whole 32-wide blocks.
__host__ __device__ inline int mm_cluster(int K) {
  for (int c = kMaxCluster; c > 1; c >>= 1)
    if (K % (32 * c) == 0) return c;
  return 1;
}

// ---------------------------------------------------------------- embedding
// x = E[token] of every sequence ("Eight kernels", decode_scale), and its sum
// of squares as the first of the nss partial sums the next RMSNorm adds up.
__global__ void __launch_bounds__(256)
    k_embed_batch(DevModel m, const DevSeq* seqs, int n, float* X, float* ss, int nss) {
  __shared__ float red[32];
  pdl_wait();  // the previous step's argmax wrote the token and the position
  pdl_launch_dependents();
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
  float acc = 0.f;
  if (m.wtype == kFmtQ8) {
    const uint8_t* row = m.embed + static_cast<size_t>(tok) * m.row_bytes_h;
    const __half* sc = reinterpret_cast<const __half*>(row + m.H);
    for (int i = threadIdx.x; i < m.H; i += blockDim.x) {
      const float v = __half2float(sc[i >> 5]) * static_cast<float>(static_cast<int8_t>(row[i]));
      x[i] = v;
      acc = fmaf(v, v, acc);
    }
  } else {
    const uint16_t* row = reinterpret_cast<const uint16_t*>(m.embed + static_cast<size_t>(tok) * m.row_bytes_h);
    for (int i = threadIdx.x; i < m.H; i += blockDim.x) {
      const float v = __uint_as_float(static_cast<uint32_t>(row[i]) << 16);
      x[i] = v;
      acc = fmaf(v, v, acc);
    }
  }
  acc = block_sum(acc, red);
  for (int i = threadIdx.x; i < nss; i += blockDim.x) ss[i * kTcN + b] = i == 0 ? acc : 0.f;
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
  pdl_wait();  // the projections of this layer are complete
  pdl_launch_dependents();
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

}  // namespace

int batch_max() { return kTcN; }

int batch_ss_slots(int H) { return ((H + kTcM - 1) / kTcM) * kMaxCluster; }

bool batch_supported(const DevModel& m) {
  const int G = m.nq / m.nkv;
  return G >= 1 && G <= 4 && (m.hd == 64 || m.hd == 128) && m.H % 64 == 0 && m.qw % 64 == 0 &&
         m.I % 64 == 0 && attn_batch_smem(m) <= 227 * 1024;
}

cudaError_t batch_setup(const DevModel& m) {
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&k_mm16),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kMmSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(&k_attn_batch),
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(attn_batch_smem(m)));
}

// One batched step for sequences seqs[0..n): embedding, every layer, lm_head
// and argmax.  X, QKV, ATTN, H are batch activations; SS holds the partial
// sums of squares of x ([slots][16]) and of x after attention (the next
// [slots][16]).  Every kernel is launched with programmatic dependent launch:
// it starts streaming its weights (or cached K/V rows) while its predecessor
// finishes, and waits for it before touching activations.
cudaError_t enqueue_batch_step(const DevModel& m, const DevLayer* host_layers, const DevSeq* seqs,
                               int n, int nch, float* X, float* QKV, float* ATTN, float* H, float* SS,
                               uint32_t* count, uint32_t* err, cudaStream_t st) {
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  auto config = [&](int grid, int threads, size_t smem, int cluster) {
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(grid);
    c.blockDim = dim3(threads);
    c.dynamicSmemBytes = smem;
    c.stream = st;
    c.attrs = at;
    c.numAttrs = 1;
    if (cluster > 1) {
      at[1].id = cudaLaunchAttributeClusterDimension;
      at[1].val.clusterDim.x = cluster;
      at[1].val.clusterDim.y = 1;
      at[1].val.clusterDim.z = 1;
      c.numAttrs = 2;
    }
    return c;
  };
  const int fmt = m.wtype;
  const int tiles_h = (m.H + kTcM - 1) / kTcM;
  float* ss_x = SS;                                       // after the embedding / down projection
  float* ss_mid = SS + batch_ss_slots(m.H) * kTcN;        // after the O projection
  const int nss_x = tiles_h * mm_cluster(m.I), nss_mid = tiles_h * mm_cluster(m.qw);
  cudaLaunchConfig_t ce = config(n, 256, 0, 1);
  cudaError_t e = cudaLaunchKernelEx(&ce, k_embed_batch, m, seqs, n, X, ss_x, nss_x);
  if (e != cudaSuccess) return e;
  auto mm = [&](const uint8_t* W, size_t rb, int K, int rows, const float* Xin, int ldx, const float* gain,
                const float* ss, int nss, int epi, float* Y, int ldy, float* ss_out, bool split) {
    MmArgs a{};
    a.W = W; a.rb = rb; a.K = K; a.rows = rows; a.fmt = fmt;
    a.cs = split ? mm_cluster(K) : 1;
    a.X = Xin; a.ldx = ldx; a.n = n; a.gain = gain; a.ss = ss; a.nss = nss; a.eps = m.eps;
    a.epi = epi; a.Y = Y; a.ldy = ldy; a.ss_out = ss_out;
    a.seqs = seqs; a.count = count; a.err = err; a.max_seq = m.max_seq;
    const int tiles = (rows + kTcM - 1) / kTcM;
    cudaLaunchConfig_t c = config(tiles * a.cs, kMmThreads, kMmSmem, a.cs);
    return cudaLaunchKernelEx(&c, k_mm16, a);
  };
  const int lqkv = m.qw + 2 * m.kvw;
  for (int l = 0; l < m.n_layers; ++l) {
    const DevLayer& L = host_layers[l];
    if ((e = mm(L.wqkv, m.row_bytes_h, m.H, lqkv, X, m.H, L.attn_norm, ss_x, nss_x, kEpiStore, QKV, lqkv,
                nullptr, true)) != cudaSuccess)
      return e;
    cudaLaunchConfig_t ca = config(n * m.nkv * nch, kAT + 32, attn_batch_smem(m), 1);
    if ((e = cudaLaunchKernelEx(&ca, k_attn_batch, m, seqs, l, nch, static_cast<const float*>(QKV), ATTN)) !=
        cudaSuccess)
      return e;
    if ((e = mm(L.wo, m.row_bytes_qw, m.qw, m.H, ATTN, m.qw, nullptr, nullptr, 0, kEpiResid, X, m.H, ss_mid,
                true)) != cudaSuccess)
      return e;
    if ((e = mm(L.wgu, m.row_bytes_h, m.H, 2 * m.I, X, m.H, L.ffn_norm, ss_mid, nss_mid, kEpiSwiGLU, H, m.I,
                nullptr, true)) != cudaSuccess)
      return e;
    if ((e = mm(L.wd, m.row_bytes_i, m.I, m.H, H, m.I, nullptr, nullptr, 0, kEpiResid, X, m.H, ss_x, true)) !=
        cudaSuccess)
      return e;
  }
  return mm(m.lm_head, m.row_bytes_h, m.H, m.V, X, m.H, m.out_norm, ss_x, nss_x, kEpiArgmax, nullptr, 0,
            nullptr, false);
}

}  // namespace tqd
