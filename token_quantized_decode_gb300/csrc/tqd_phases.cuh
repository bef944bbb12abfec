// The phases of one decode step as device functions over a (block, nblocks)
// work split, so the same code runs as one kernel per phase (CUDA-graph
// schedule), inside the persistent kernel, and behind the operator entry
// points.
//
// What each phase computes follows the inferno.rs blog, "IV.4: One command
// buffer per token", section "Eight kernels" (q8_matvec, rms_norm_row,
// rope_row, append_kv, attention_decode, add_inplace, silu_hadamard,
// argmax_row) in the op order of section "One command buffer".
#pragma once

#include "tqd_device.cuh"

namespace tqd {


// SwiGLU gate: silu(g) * u with silu(z) = z / (1 + e^-z) ("Eight kernels",
// silu_hadamard).
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// ---------------------------------------------------------------------------
// block-wide helpers
// ---------------------------------------------------------------------------
// Sum over the block; `red` is >= 32 floats of shared memory.  Every thread
// gets the total.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += red[i];
  return t;
}

// Stage n floats (n * 4 a multiple of 16, both addresses 16-byte aligned)
// from global memory into shared memory with one bulk copy issued by thread
// 0; every thread waits on the mbarrier.  The caller must have finished all
// reads of dst (a __syncthreads) before calling.
__device__ __forceinline__ bool stage_vector(float* dst, const float* src, int n, uint64_t* bar,
                                             uint32_t& parity, uint32_t* err) {
  if (threadIdx.x == 0) {
    fence_proxy_async_global();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n) * 4u);
    bulk_g2s(dst, src, static_cast<uint32_t>(n) * 4u, bar);
  }
  const bool ok = mbar_wait_bounded(bar, parity, err);
  parity ^= 1u;
  return ok;
}

// xs[i] <- xs[i] * (mean(xs^2) + eps)^(-1/2) * g[i]   ("Eight kernels",
// rms_norm_row: sum of squares, reciprocal square root, gain).
__device__ __forceinline__ void rmsnorm_smem(float* xs, const float* g, int n, float eps,
                                             float* red) {
  float ss = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) ss = fmaf(xs[i], xs[i], ss);
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / static_cast<float>(n) + eps);
  for (int i = threadIdx.x; i < n; i += blockDim.x) xs[i] = xs[i] * inv * __ldg(g + i);
  __syncthreads();
}

// ---------------------------------------------------------------------------
// matvec core: one warp, R consecutive rows, K columns, x in shared memory.
// Lane l owns the 16-byte chunks l, l+32, ... of each row: coalesced 128-bit
// loads of the quants (Q8_0 row layout: K int8 then K/32 f16 scales), one
// scale per half block.  acc[rr] returns the lane's partial dot product.
// ---------------------------------------------------------------------------
template <int FMT, int CPL, int R>
__device__ __forceinline__ void matvec_rows(const uint8_t* __restrict__ W, size_t row_bytes, int K,
                                            int r0, int rows_end, const float* __restrict__ xs,
                                            float (&acc)[R]) {
  const int lane = threadIdx.x & 31;
  constexpr int EPC = (FMT == kFmtQ8) ? 16 : 8;  // weights per 16-byte chunk
  const int nchunks = K / EPC;
  uint4 wv[R][CPL];
  uint16_t sv[R][CPL];
#pragma unroll
  for (int rr = 0; rr < R; ++rr) {
    const int r = r0 + rr;
    const uint8_t* row = W + static_cast<size_t>(r) * row_bytes;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      if (r < rows_end && c < nchunks) {
        wv[rr][i] = ld_weights16(row + 16 * c);
        if (FMT == kFmtQ8) sv[rr][i] = ld_weights_u16(row + K + 2 * (c >> 1));
      } else {
        wv[rr][i] = make_uint4(0u, 0u, 0u, 0u);
        sv[rr][i] = 0;
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < R; ++rr) acc[rr] = 0.f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = lane + 32 * i;
    if (c < nchunks) {
      float xv[EPC];
      const float4* xp = reinterpret_cast<const float4*>(xs + EPC * c);
#pragma unroll
      for (int k = 0; k < EPC / 4; ++k) {
        const float4 t = xp[k];
        xv[4 * k] = t.x;
        xv[4 * k + 1] = t.y;
        xv[4 * k + 2] = t.z;
        xv[4 * k + 3] = t.w;
      }
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const uint32_t w4[4] = {wv[rr][i].x, wv[rr][i].y, wv[rr][i].z, wv[rr][i].w};
        if (FMT == kFmtQ8) {
          float p0 = 0.f, p1 = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float a, b, c2, d;
            i8x4_to_f32(w4[k], a, b, c2, d);
            p0 = fmaf(a, xv[4 * k], p0);
            p1 = fmaf(b, xv[4 * k + 1], p1);
            p0 = fmaf(c2, xv[4 * k + 2], p0);
            p1 = fmaf(d, xv[4 * k + 3], p1);
          }
          const float s = __half2float(__ushort_as_half(sv[rr][i]));
          acc[rr] = fmaf(s, p0 + p1, acc[rr]);
        } else {
          float p0 = 0.f, p1 = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            p0 = fmaf(bf16_lo(w4[k]), xv[2 * k], p0);
            p1 = fmaf(bf16_hi(w4[k]), xv[2 * k + 1], p1);
          }
          acc[rr] += p0 + p1;
        }
      }
    }
  }
}

// Rows per warp group for a chunk count per lane: enough loads in flight per
// lane (R * CPL 16-byte chunks), and an even count so gate/up pairs stay in
// one warp.
template <int CPL>
struct RowsPerGroup {
  static constexpr int value = (8 / CPL) >= 2 ? (8 / CPL) : 2;
};

struct MatvecJob {
  const uint8_t* W;
  size_t row_bytes;
  int K;
  int rows;        // matrix rows
  int epi;         // kEpi*
  float* y;        // output (store / residual target / SwiGLU output / logits)
};

// Per-warp running argmax of the lm_head epilogue.
struct ArgmaxAcc {
  float v;
  int i;
};

// All row groups of a matrix split over the warps of blocks [0, nblocks).
template <int FMT, int CPL>
__device__ __forceinline__ void matvec_phase(const MatvecJob& job, const float* xs, int block,
                                             int nblocks, ArgmaxAcc& am) {
  constexpr int R = RowsPerGroup<CPL>::value;
  const int lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int gw = block * nw + (threadIdx.x >> 5);
  const int stride = nblocks * nw;
  const int ngroups = (job.rows + R - 1) / R;
  for (int grp = gw; grp < ngroups; grp += stride) {
    const int r0 = grp * R;
    float acc[R];
    matvec_rows<FMT, CPL, R>(job.W, job.row_bytes, job.K, r0, job.rows, xs, acc);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) acc[rr] = warp_sum(acc[rr]);
    if (lane == 0) {
      if (job.epi == kEpiSwiGLU) {
#pragma unroll
        for (int rr = 0; rr + 1 < R; rr += 2) {
          const int r = r0 + rr;
          if (r + 1 < job.rows) {
            job.y[r >> 1] = silu_mul(acc[rr], acc[rr + 1]);
          }
        }
      } else {
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
          const int r = r0 + rr;
          if (r < job.rows) {
            if (job.epi == kEpiStore) {
              job.y[r] = acc[rr];
            } else if (job.epi == kEpiResid) {
              job.y[r] = ld_cg(job.y + r) + acc[rr];
            } else {
              job.y[r] = acc[rr];
              argmax_merge(am.v, am.i, acc[rr], r);
            }
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// argmax: reduce per-warp candidates to one per block, publish it, and let
// the last block to arrive reduce all blocks' candidates.  Returns true in
// the last block (all threads), with the winner in (*win_v, *win_i).
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool argmax_blocks(ArgmaxAcc am, int block, int nblocks, float* cand_v,
                                              int32_t* cand_i, uint32_t* count, float* red,
                                              float* win_v, int* win_i) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int* redi = reinterpret_cast<int*>(red + 32);
  __shared__ uint32_t s_last;
  // lane 0 of each warp holds its warp's candidate
  __syncthreads();
  if (lane == 0) {
    red[warp] = am.v;
    redi[warp] = am.i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int w = 0; w < nw; ++w) argmax_merge(bv, bi, red[w], redi[w]);
    cand_v[block] = bv;
    cand_i[block] = bi;
    __threadfence();
    const uint32_t old = atomicAdd(count, 1u);
    s_last = (old == static_cast<uint32_t>(nblocks) - 1u) ? 1u : 0u;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return false;
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  for (int b = threadIdx.x; b < nblocks; b += blockDim.x)
    argmax_merge(bv, bi, __ldcg(cand_v + b), __ldcg(cand_i + b));
  warp_argmax(bv, bi);
  __syncthreads();
  if (lane == 0) {
    red[warp] = bv;
    redi[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = -INFINITY;
    int i = 0x7FFFFFFF;
    for (int w = 0; w < nw; ++w) argmax_merge(v, i, red[w], redi[w]);
    *win_v = v;
    *win_i = i;
    *count = 0u;  // ready for the next use
  }
  __syncthreads();
  return true;
}

// ---------------------------------------------------------------------------
// attention: split-K flash decode ("Eight kernels", attention_decode, with
// the score row replaced by an online softmax over key chunks and a
// log-sum-exp combine of the chunks).
// ---------------------------------------------------------------------------
struct AttnJob {
  const float* q;        // [nq*HD] query (raw when q_norm / rope given)
  const float* k_new;    // [nkv*HD] raw k of the new row, or nullptr (no append)
  const float* v_new;
  const float* q_norm;   // [HD] or nullptr
  const float* k_norm;
  const float2* rope;    // (cos, sin) row of the current position, or nullptr
  float* kc;             // keys of this layer (post-RoPE): row t of kv head g at
  float* vc;             //   kc + g * head_stride + t * row_stride (in elements)
  size_t head_stride, row_stride;
  int kv16;              // the cache holds f16 elements (kc, vc point at halves)
  int S, nq, nkv, n_chunks;
  float eps, scale;
  float* part_o;         // [nq][n_chunks][HD]
  float* part_ml;        // [nq][n_chunks][2]
  uint32_t* count;       // [nkv], zero between uses
  float* out;            // [nq*HD]
};

// Shared memory needed by attention_item (floats).
__host__ __device__ constexpr int attn_smem_floats(int hd, int G, int nwarps) {
  return G * hd + nwarps * G * (hd + 2) + 64;
}

// Normalise (optional) and rotate (optional) one head held as lane-strided
// elements e_j = lane + 32 j.
template <int HD>
__device__ __forceinline__ void head_norm_rope(float (&v)[HD / 32], const float* gain,
                                               const float2* rope, float eps) {
  const int lane = threadIdx.x & 31;
  constexpr int NJ = HD / 32;
  if (gain) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) ss = fmaf(v[j], v[j], ss);
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / static_cast<float>(HD) + eps);
#pragma unroll
    for (int j = 0; j < NJ; ++j) v[j] = v[j] * inv * __ldg(gain + lane + 32 * j);
  }
  if (rope) {
    // pair (i, i + HD/2): i = lane + 32 j for j < NJ/2
#pragma unroll
    for (int j = 0; j < NJ / 2; ++j) {
      const float2 cs = __ldg(rope + lane + 32 * j);
      const float u = v[j], w = v[j + NJ / 2];
      v[j] = u * cs.x - w * cs.y;
      v[j + NJ / 2] = u * cs.y + w * cs.x;
    }
  }
}

template <int HD, int G>
__device__ void attention_item(const AttnJob& a, int g, int c, float* smem, uint32_t* err) {
  constexpr int DPL = HD / 32;  // contiguous elements per lane in the key scan
  constexpr int NJ = HD / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float* qs = smem;                      // [G][HD]
  float* wst = smem + G * HD;            // [nw][G][HD + 2]
  __shared__ uint32_t s_last;
  const int S = a.S;
  const int cs = (S + a.n_chunks - 1) / a.n_chunks;
  const int t0 = min(S, c * cs), t1 = min(S, t0 + cs);
  const int pos = S - 1;

  // 1. queries of this kv group: norm + RoPE into shared memory
  for (int hh = warp; hh < G; hh += nw) {
    const int h = g * G + hh;
    float v[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) v[j] = ld_cg(a.q + h * HD + lane + 32 * j);
    head_norm_rope<HD>(v, a.q_norm, a.rope, a.eps);
#pragma unroll
    for (int j = 0; j < NJ; ++j) qs[hh * HD + lane + 32 * j] = v[j];
  }
  // 2. the chunk holding the new position appends its K/V row ("Eight
  //    kernels", append_kv) before scanning it
  if (a.k_new != nullptr && t0 <= pos && pos < t1 && warp == 0) {
    float kv[NJ], vv[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      kv[j] = ld_cg(a.k_new + g * HD + lane + 32 * j);
      vv[j] = ld_cg(a.v_new + g * HD + lane + 32 * j);
    }
    head_norm_rope<HD>(kv, a.k_norm, a.rope, a.eps);
    const size_t off = g * a.head_stride + static_cast<size_t>(pos) * a.row_stride;
    if (a.kv16) {  // rounded to binary16 as the row enters the cache; the scan reads it back
      __half* krow = reinterpret_cast<__half*>(a.kc) + off;
      __half* vrow = reinterpret_cast<__half*>(a.vc) + off;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        krow[lane + 32 * j] = __float2half_rn(kv[j]);
        vrow[lane + 32 * j] = __float2half_rn(vv[j]);
      }
    } else {
      float* krow = a.kc + off;
      float* vrow = a.vc + off;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        krow[lane + 32 * j] = kv[j];
        vrow[lane + 32 * j] = vv[j];
      }
    }
  }
  __syncthreads();

  // 3. online softmax over this chunk's rows, one warp per row
  float m[G], l[G], o[G][DPL];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    m[hh] = -INFINITY;
    l[hh] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[hh][d] = 0.f;
  }
  float qv[G][DPL];
#pragma unroll
  for (int hh = 0; hh < G; ++hh)
#pragma unroll
    for (int d = 0; d < DPL; ++d) qv[hh][d] = qs[hh * HD + lane * DPL + d];

  for (int t = t0 + warp; t < t1; t += nw) {
    const size_t off = g * a.head_stride + static_cast<size_t>(t) * a.row_stride + lane * DPL;
    const float* krow = a.kc + off;
    const float* vrow = a.vc + off;
    float kf[DPL], vf[DPL];
    if (a.kv16) {
      const __half* kh = reinterpret_cast<const __half*>(a.kc) + off;
      const __half* vh = reinterpret_cast<const __half*>(a.vc) + off;
#pragma unroll
      for (int e = 0; e < DPL; e += 2) {
        const float2 k2 = __half22float2(__ldcg(reinterpret_cast<const __half2*>(kh + e)));
        const float2 v2 = __half22float2(__ldcg(reinterpret_cast<const __half2*>(vh + e)));
        kf[e] = k2.x; kf[e + 1] = k2.y;
        vf[e] = v2.x; vf[e + 1] = v2.y;
      }
    } else if constexpr (DPL == 4) {
      const float4 k4 = ld_cg4(reinterpret_cast<const float4*>(krow));
      const float4 v4 = ld_cg4(reinterpret_cast<const float4*>(vrow));
      kf[0] = k4.x; kf[1] = k4.y; kf[2] = k4.z; kf[3] = k4.w;
      vf[0] = v4.x; vf[1] = v4.y; vf[2] = v4.z; vf[3] = v4.w;
    } else {
      const float2 k2 = ld_cg2(reinterpret_cast<const float2*>(krow));
      const float2 v2 = ld_cg2(reinterpret_cast<const float2*>(vrow));
      kf[0] = k2.x; kf[1] = k2.y;
      vf[0] = v2.x; vf[1] = v2.y;
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) d = fmaf(qv[hh][e], kf[e], d);
      const float s = warp_sum(d) * a.scale;
      if (s > m[hh]) {
        const float corr = expf(m[hh] - s);
        m[hh] = s;
        l[hh] = l[hh] * corr + 1.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[hh][e] = fmaf(o[hh][e], corr, vf[e]);
      } else {
        const float p = expf(s - m[hh]);
        l[hh] += p;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[hh][e] = fmaf(p, vf[e], o[hh][e]);
      }
    }
  }
  // 4. merge the warps of this block, write the chunk's partial
  const int stride = HD + 2;
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    float* w = wst + (warp * G + hh) * stride;
#pragma unroll
    for (int e = 0; e < DPL; ++e) w[lane * DPL + e] = o[hh][e];
    if (lane == 0) {
      w[HD] = m[hh];
      w[HD + 1] = l[hh];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * HD; idx += blockDim.x) {
    const int hh = idx / HD, d = idx - hh * HD;
    float M = -INFINITY;
    for (int w = 0; w < nw; ++w) M = fmaxf(M, wst[(w * G + hh) * stride + HD]);
    float O = 0.f, L = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < nw; ++w) {
        const float* ws = wst + (w * G + hh) * stride;
        const float f = expf(ws[HD] - M);  // 0 for warps that saw no row
        O = fmaf(f, ws[d], O);
        L = fmaf(f, ws[HD + 1], L);
      }
    }
    const int h = g * G + hh;
    a.part_o[(static_cast<size_t>(h) * a.n_chunks + c) * HD + d] = O;
    if (d == 0) {
      a.part_ml[(static_cast<size_t>(h) * a.n_chunks + c) * 2] = M;
      a.part_ml[(static_cast<size_t>(h) * a.n_chunks + c) * 2 + 1] = L;
    }
  }
  // 5. the last chunk of this kv group to finish combines all chunks
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(a.count + g, 1u);
    s_last = (old == static_cast<uint32_t>(a.n_chunks) - 1u) ? 1u : 0u;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  for (int idx = threadIdx.x; idx < G * HD; idx += blockDim.x) {
    const int hh = idx / HD, d = idx - hh * HD;
    const int h = g * G + hh;
    const float* ml = a.part_ml + static_cast<size_t>(h) * a.n_chunks * 2;
    const float* po = a.part_o + static_cast<size_t>(h) * a.n_chunks * HD;
    float M = -INFINITY;
    for (int cc = 0; cc < a.n_chunks; ++cc) M = fmaxf(M, __ldcg(ml + 2 * cc));
    float num = 0.f, den = 0.f;
    for (int cc = 0; cc < a.n_chunks; ++cc) {
      const float mc = __ldcg(ml + 2 * cc);
      if (mc == -INFINITY) continue;
      const float f = expf(mc - M);
      num = fmaf(f, __ldcg(po + static_cast<size_t>(cc) * HD + d), num);
      den = fmaf(f, __ldcg(ml + 2 * cc + 1), den);
    }
    a.out[h * HD + d] = num / den;
  }
  __syncthreads();
  if (threadIdx.x == 0) a.count[g] = 0u;
  (void)err;
}

}  // namespace tqd
