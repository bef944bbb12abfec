// Device-side building blocks for the decode kernels: inline-PTX wrappers
// (mbarrier, 1-D bulk TMA copies, proxy fences, programmatic dependent
// launch, acquire/release), bounded waits that report instead of hanging,
// int8 -> f32 conversion, warp reductions, and the device model layout.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace tqd {

// ---------------------------------------------------------------------------
// error word bits (DevState::err); the host turns them into statuses
// ---------------------------------------------------------------------------
enum : uint32_t {
  kErrGridBarrier = 1u,   // a grid barrier wait ran out of time
  kErrMbarrier = 2u,      // an mbarrier (bulk copy) wait ran out of time
  kErrAllNaN = 4u,        // every logit was NaN
  kErrBadToken = 8u,      // a token id outside [0, vocab)
  kErrCapacity = 16u,     // a position at or beyond max_seq
};

// weight formats and matvec epilogues
enum { kFmtQ8 = 0, kFmtBF16 = 1 };
enum { kEpiStore = 0, kEpiResid = 1, kEpiSwiGLU = 2, kEpiArgmax = 3, kEpiTagged = 4, kEpiAtomicAdd = 5 };

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier + 1-D bulk copy (TMA without a tensor map)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of the barrier to complete; false (and the error
// bit set) if it does not within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      if (err) atomicOr(err, kErrMbarrier);
      return false;
    }
  }
  return true;
}

// Global -> shared bulk copy completing on `bar` (both addresses 16-byte
// aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// An L2 policy that marks lines as the first to evict: for the weight and K/V
// streams, read once per step, so that they do not push the small data every
// step re-reads (norm gains, RoPE rows, activations) out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Order this thread's generic-proxy global accesses with later async-proxy
// (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// loads / stores with explicit cache behaviour
// ---------------------------------------------------------------------------
// Weights: read once per step, never written -> non-coherent path, no L1 fill.
__device__ __forceinline__ uint4 ld_weights16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint16_t ld_weights_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Data another CTA of the same launch may have written: L2 only.
__device__ __forceinline__ float ld_cg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float4 ld_cg4(const float4* p) { return __ldcg(p); }
__device__ __forceinline__ float2 ld_cg2(const float2* p) { return __ldcg(p); }

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_u32(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

// ---------------------------------------------------------------------------
// int8 x4 -> f32 x4, exact: byte b -> (b ^ 0x80) = q + 128 placed in the low
// mantissa bits of 2^23, then 2^23 + 128 subtracted.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float& f0, float& f1, float& f2,
                                            float& f3) {
  const uint32_t t = w ^ 0x80808080u;
  f0 = __uint_as_float(__byte_perm(t, 0x4B000000u, 0x7640)) - 8388736.0f;
  f1 = __uint_as_float(__byte_perm(t, 0x4B000000u, 0x7641)) - 8388736.0f;
  f2 = __uint_as_float(__byte_perm(t, 0x4B000000u, 0x7642)) - 8388736.0f;
  f3 = __uint_as_float(__byte_perm(t, 0x4B000000u, 0x7643)) - 8388736.0f;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// (value, index) argmax step: larger value wins, ties -> lower index, NaN
// never wins (a NaN candidate fails both comparisons).
__device__ __forceinline__ void argmax_merge(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}
__device__ __forceinline__ void warp_argmax(float& bv, int& bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
    int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
    argmax_merge(bv, bi, ov, oi);
  }
}

// ---------------------------------------------------------------------------
// the device model
// ---------------------------------------------------------------------------
// Q8_0 matrices are stored row-repacked: each row of K weights is K int8
// quants followed by K/32 f16 scales, padded to a multiple of 16 bytes
// (K*17/16 bytes, no padding, when K % 256 == 0).  bf16 matrices are plain row-major.  Q, K and V projection
// rows are concatenated into one [qw + 2 kvw] x H matrix; gate and up rows are
// interleaved (row 2j = gate j, row 2j+1 = up j) into one [2I] x H matrix.
struct DevLayer {
  const uint8_t* wqkv;
  const uint8_t* wo;
  const uint8_t* wo_g;    // persistent schedule: wo's columns split by kv group, [n_kv][H][G hd]
  const uint8_t* wgu;
  const uint8_t* wd;
  const uint8_t* wd_c;    // persistent schedule: wd by column blocks (see DevModel::dcol_bytes)
  const float* attn_norm;
  const float* q_norm;
  const float* k_norm;
  const float* ffn_norm;
};

struct DevState {  // per sequence, in device memory
  uint32_t pos;    // next position (= KV rows filled)
  uint32_t err;    // kErr* bits
  uint32_t steps;  // steps completed (diagnostic)
  int32_t last;    // the token the last greedy step wrote at its next position (-1: every logit NaN)
};

// Barrier of the persistent schedule (the whole grid, or the blocks of one kv
// group): a monotonic arrival count and the number of barriers completed so
// far.  Set to zero once at creation and never reset, so every barrier's
// target is (completed + 1) * members.
struct DevBarrier {
  unsigned long long count;
  unsigned long long epoch;
};

struct DevModel {
  int n_layers, H, nq, nkv, hd, I, V, qk_norm, wtype, max_seq;
  int qw, kvw, n_chunks;  // n_chunks: split-K chunks of the attention
  float eps, attn_scale;
  size_t row_bytes_h;     // bytes per row of a matrix with H columns
  size_t row_bytes_qw;    // ... with qw columns
  size_t row_bytes_i;     // ... with I columns
  size_t row_bytes_gh;    // ... with (n_heads / n_kv_heads) * head_dim columns
  // The down projection by columns (persistent schedule), so that a block that
  // owns SwiGLU outputs h[j0, j1) reads exactly the columns that multiply them.
  // Q8_0: per 32-column block c, the H f16 scales of that block's rows (padded
  // to 16 bytes), then 32 runs of H int8 quants, run j the quants of column
  // 32c + j for rows 0..H-1; dcol_bytes is the size of one such block.  bf16:
  // per column j, its H values; dcol_bytes = 2H.
  size_t dcol_bytes;
  const DevLayer* layers;
  const uint8_t* lm_head;
  const uint8_t* embed;
  const float* out_norm;
  const float2* rope;     // [max_seq][hd/2] (cos, sin)
  int kv16;               // the KV cache holds f16 elements (the batched kernels only)
};

// Per-sequence buffers.
struct DevSeq {
  DevState* state;
  int32_t* tokens;        // [max_seq + 1]: input token of each position
  float* kcache;          // [n_layers][n_kv_heads][max_seq][head_dim] (f16 elements when kv16)
  float* vcache;
  float* x;               // [H] residual stream
  float* qkv;             // [qw + 2 kvw] raw projections
  float* attn;            // [qw] attention output
  float* h;               // [I] SwiGLU output
  float* logits;          // [V]
  float* part_o;          // [nq][n_chunks][hd]
  float* part_ml;         // [nq][n_chunks][2]
  uint32_t* attn_count;   // [nkv] arrivals per kv head
  float* amax_v;          // [max_ctas] per-CTA argmax candidates
  int32_t* amax_i;
  uint32_t* amax_count;   // [1]
  DevBarrier* bar;        // grid barrier of the persistent schedule
  float* x_mid;           // [H] residual after the attention block
  DevBarrier* gbar;       // per kv group g: [16 g] QKV rows written, [16 g + 8] attention partials written
  float* opart;           // [2][H] the persistent schedule's O products, summed over groups (two sets)
  float* sz;              // [V] the sampler's penalised logits
  uint32_t* scnt;         // [V] the sampler's input-token counts (zero between draws)
  float* xacc;            // [2][4][H] the persistent schedule's down-projection sums (two sets of four copies)
  uint64_t* qkv_tag;      // [qw + 2 kvw] the persistent schedule's projections as (tag << 32 | f32 bits) words
  unsigned long long* sparts;  // the sampler's per-slice top_k keys [ceil(V / 1024)][64], or null
  int32_t tok_in;         // persistent schedule: the first step's input token when >= 0 (the kernel
                          // stores it at tokens[pos]); -1: the token is already at tokens[pos]
};

}  // namespace tqd
