// Batched decode step: up to 16 sequences advance one token together, so
// every projection is a dense [rows x K] x [K x n] contraction that runs on the
// fifth-generation tensor cores (tcgen05, accumulator in tensor memory), and
// attention runs per sequence as a streaming split-K flash decode.
//
// Numerics (kind::f16, f32 accumulation): a Q8_0 quant is an integer in
// [-127, 127], exact in bf16 and in f16, so the weights enter as A unchanged;
// every 32-wide block accumulates into its own tensor-memory columns and its
// f16 scale multiplies the block's sums at read-out.  The activations enter as
// B split into parts: three bf16 parts in the projections (24 significant
// bits: each product is exact and the sums are f32 sums), two f16 parts in the
// lm_head, whose input is the bounded RMSNorm output (22 significant bits).
// bf16 weights are exact in bf16 (scale 1); the lm_head stores them as f16.
//
// What is computed is the decode step of the inferno.rs blog, "IV.4: One
// command buffer per token", for several sequences sharing one sweep of the
// weights ("Metal LLM decode", the batched prefill+decode arm).
#include <algorithm>
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
constexpr int kTcN = 16;               // batch rows
constexpr int kTcN3 = 3 * kTcN;        // MMA N: the three bf16 parts of every batch row
constexpr int kSubK = 64;              // K elements per A / B sub-chunk
constexpr int kPassBytes = 128;        // weight bytes per row per pass (Q8_0: 128 K, bf16: 64 K)
constexpr uint32_t kRawBytes = kTcM * kPassBytes;    // one raw stage; 16-byte chunks XOR-swizzled per row
constexpr uint32_t kABytes = kTcM * kSubK * 2;       // one bf16 A sub-chunk
constexpr uint32_t kAPassBytes = 2 * kABytes;        // A of one pass (up to 128 K)
constexpr uint32_t kBPartBytes = kTcN * kSubK * 2;   // one bf16 part of B
constexpr uint32_t kBBytes = 3 * kBPartBytes;        // one sub-chunk of B: N = 48 rows
constexpr int kMaxCluster = 16;       // 16 is a non-portable cluster size (allowed per kernel)
// rows of a tile each cluster rank reduces: whole row pairs, split as evenly as
// the cluster size allows (at most 2 * ceil(64 / cs) rows)
__host__ __device__ constexpr int pair_row0(int q, int cs) { return 2 * ((q * (kTcM / 2)) / cs); }
__host__ __device__ constexpr int recv_stride(int cs) { return 2 * ((kTcM / 2 + cs - 1) / cs); }
constexpr int kRecvRows = 160;       // >= cs * recv_stride(cs) for every cs <= 16
// Shared memory of a split projection CTA (one tile, two CTAs per SM): raw
// weight stages, one pass of A, B for up to MAXSUB sub-chunks (384 K), and
// the partial sums received from the cluster ranks.
template <int STAGES, int MAXSUB>
struct MmCfg {
  static constexpr int threads = kMmThreads;
  static constexpr uint32_t a = STAGES * kRawBytes;
  static constexpr uint32_t b = a + kAPassBytes;
  static constexpr uint32_t recv = b + MAXSUB * kBBytes;
  static constexpr uint32_t total = recv + kRecvRows * kTcN * 4;  // [rank][row][16] partials received
  static constexpr uint32_t tmem = 256;                          // one pass: four blocks of 48 columns
};
using SplitCfg = MmCfg<2, 6>;
static_assert(2 * (SplitCfg::total + 2048) <= 228 * 1024, "two split CTAs per SM");
constexpr int kSplitMaxK = 6 * kSubK, kHeadMaxK = 16 * kSubK;  // K of a split rank, of the lm_head

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

// kind::f16 with f16 A and B, f32 accumulator, both K-major, shape M x N.
constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr int kHdN = 2 * kTcN;  // the lm_head's MMA N: two f16 parts of every batch row
__device__ __forceinline__ void mma_f16_hd(uint32_t dt, uint64_t ad, uint64_t bd, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dt),
      "l"(ad), "l"(bd), "r"(idesc_f16(kTcM, kHdN)), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t dt, uint64_t ad, uint64_t bd, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dt),
      "l"(ad), "l"(bd), "r"(idesc_bf16(kTcM, kTcN3)), "r"(acc)
      : "memory");
}

// The MMAs of one pass: nb 32-wide blocks, two K = 16 steps each, block blk
// into accumulator columns d + blk * n.  da / db are the descriptors of the
// pass's A and of its first B sub-chunk; a descriptor's address field is the
// byte address / 16 (shared memory stays below 256 KB, so adding an offset
// / 16 never carries out of the field).  With nb == 4 (a full pass) the loop
// is unrolled to constant offsets: one thread issues these, so its
// instruction count per MMA is on the critical path.
template <bool F16>
__device__ __forceinline__ void mma_pass(uint32_t d, int n, uint64_t da, uint64_t db, uint32_t bsub, int nb) {
  auto one = [&](int blk, int ks) {
    const uint32_t koff = (blk >> 1) * kABytes + ((blk & 1) * 2 + ks) * 256;  // 16 K = two core matrices
    const uint32_t boff = (blk >> 1) * bsub + ((blk & 1) * 2 + ks) * 256;
    if (F16) mma_f16_hd(d + blk * n, da + (koff >> 4), db + (boff >> 4), ks ? 1u : 0u);
    else mma_bf16(d + blk * n, da + (koff >> 4), db + (boff >> 4), ks ? 1u : 0u);
  };
  if (nb == 4) {
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      one(blk, 0);
      one(blk, 1);
    }
  } else {
    for (int blk = 0; blk < nb; ++blk) {
      one(blk, 0);
      one(blk, 1);
    }
  }
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

// Four int8 (one word) -> four f16 (two words), exact: the byte plus 128 is
// placed in the mantissa of 1024 (f16 0x64xx), and 1152 is subtracted.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t t = w ^ 0x80808080u;
  const __half2 bias = __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6480u)));
  uint32_t l = __byte_perm(t, 0x64646464u, 0x4140), h = __byte_perm(t, 0x64646464u, 0x4342);
  const __half2 hl = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
  const __half2 hh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
  lo = *reinterpret_cast<const uint32_t*>(&hl);
  hi = *reinterpret_cast<const uint32_t*>(&hh);
}

// x = x1 + x2 + r, each part f16, |r| <= 2^-22 |x| while 2^-3 <= |x| < 65504
// (below, |r| <= 2^-25: the second part reaches the f16 subnormals).
__device__ __forceinline__ void split2_f16(float x, uint32_t& p1, uint32_t& p2) {
  const __half h1 = __float2half_rn(x);
  p1 = __half_as_ushort(h1);
  p2 = __half_as_ushort(__float2half_rn(x - __half2float(h1)));
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
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void tmem_ld16(uint32_t addr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(addr)
      : "memory");
}
// The 48 columns of one block (three parts x 16 batch rows), summed per row.
__device__ __forceinline__ void tmem_block_sum(uint32_t addr, float (&v)[16]) {
  uint32_t r0[16], r1[16], r2[16];
  tmem_ld16(addr, r0);
  tmem_ld16(addr + 16, r1);
  tmem_ld16(addr + 32, r2);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = (__uint_as_float(r0[i]) + __uint_as_float(r1[i])) + __uint_as_float(r2[i]);
}
__device__ __forceinline__ void st_dsmem4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
// 16 bytes into another CTA's shared memory, counted on that CTA's mbarrier
// (both addresses from mapa)
__device__ __forceinline__ void st_async4(uint32_t addr, uint32_t bar, float a, float b, float c, float d) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ uint32_t mapa_u32(const void* p, uint32_t cta) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(cta));
  return a;
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
  int out0;             // kEpiArgmax: the first batch row whose logits and next token are kept
  uint32_t* err;
  int max_seq;
  // X given as split-K attention partials instead (nullptr: plain X): per
  // sequence b, head h and chunk c, part_o[((b * K / hd + h) * nch + c) * hd + d]
  // and part_ml[((b * K / hd + h) * nch + c) * 2 + {0, 1}] = (max, sum)
  const float* part_o;
  const float* part_ml;
  int nch, hd;
  // the next kernel's weights, prefetched into L2 before the dependency wait
  // (its CTAs that start only as this kernel ends then find them there)
  const uint8_t* pf;
  size_t pf_bytes;
};

// This CTA's share of an L2 prefetch of [p, p + bytes), 128-byte lines.
__device__ __forceinline__ void prefetch_share(const uint8_t* p, size_t bytes, int nt) {
  if (!p) return;
  const size_t lines = bytes >> 7, stride = static_cast<size_t>(gridDim.x) * nt;
  for (size_t i = static_cast<size_t>(blockIdx.x) * nt + threadIdx.x; i < lines; i += stride)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p + (i << 7)));
}

// Thread t of the CTA works on weight row t of its tile (tensor-memory lane
// t); the cluster's ranks split the tile's K, and each rank owns a range of
// the tile's row pairs for the reduction and the epilogue.
template <class CFG>
__global__ void __launch_bounds__(CFG::threads, 1) k_mm16(MmArgs a) {
  constexpr int STAGES = CFG::a / kRawBytes;
  constexpr int NT = CFG::threads, NW = NT / 32;
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ __align__(8) uint64_t bars[2];  // a pass's MMAs are complete (by pass parity)
  __shared__ __align__(8) uint64_t rbar;     // every cluster rank's partials of this CTA's rows have landed
  __shared__ uint32_t tmem_base;
  __shared__ float inv_rms[kTcN];
  __shared__ float wred_v[NW][kTcN];
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int tr = t;  // the weight row of the tile
  const int rank = static_cast<int>(cluster_rank());
  const bool q8 = a.fmt == kFmtQ8;
  // this rank's K range: whole 32-wide blocks, split as evenly as the cluster size allows
  const int nbk = a.K / 32;
  const int kc0 = 32 * ((rank * nbk) / a.cs), KR = 32 * (((rank + 1) * nbk) / a.cs) - kc0;
  const int PK = q8 ? kPassBytes : kPassBytes / 2;  // K per pass
  const int npass = (KR + PK - 1) / PK;
  const int tile = static_cast<int>(blockIdx.x) / a.cs;  // the cluster's tile
  const int total = npass;                               // passes of this CTA
  // weight quants of pass g for all 128 rows -> raw stage g % STAGES
  auto issue_raw = [&](int g) {
    const int row0 = tile * kTcM;
    const int k0 = kc0 + g * PK, pk = min(PK, kc0 + KR - k0);
    const int chunks = (q8 ? pk : 2 * pk) / 16;
    unsigned char* dst = sm + (g % STAGES) * kRawBytes;
    for (int c = t; c < kTcM * 8; c += NT) {
      const int r = c >> 3, ch = c & 7;
      if (ch < chunks) {
        const bool ok = row0 + r < a.rows;
        const uint8_t* src = a.W + static_cast<size_t>(ok ? row0 + r : 0) * a.rb + (q8 ? k0 : 2 * k0) + ch * 16;
        cp_async16(dst + r * kPassBytes + ((ch ^ (r & 7)) << 4), src, ok);
      }
    }
    cp_async_commit();
  };
  // f16 scale bits of this thread's row for the blocks of pass g
  auto load_scales = [&](int g, uint16_t (&sb)[4]) {
    const int row = tile * kTcM + tr;
    const int k0 = kc0 + g * PK, nblk = min(PK, kc0 + KR - k0) / 32;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      sb[i] = (q8 && g < total && row < a.rows && i < nblk)
                  ? ld_weights_u16(a.W + static_cast<size_t>(row) * a.rb + a.K + 2 * (k0 / 32 + i))
                  : static_cast<uint16_t>(0);
  };
  // split-K over a cluster: every rank sends its partial sums of the rows
  // rank q owns straight into q's shared memory with st.async, and q waits on
  // rbar for all of them (no cluster-wide barrier after the MMAs); rows
  // [own0, own0 + own) of the tile are this rank's
  const bool push = a.cs > 1;
  const int own0 = pair_row0(rank, a.cs), own = pair_row0(rank + 1, a.cs) - own0;
  // weights never depend on earlier kernels: their loads are issued first,
  // before the dependency wait and before the setup below, whose latency they
  // then overlap (a CTA that starts only as the previous kernel ends would
  // otherwise pay both)
  for (int g = 0; g < STAGES - 1; ++g) {
    if (g < total) issue_raw(g);
    else cp_async_commit();  // empty groups keep the group count uniform
  }
  // block scales of the next two passes, loaded as far ahead as their quants
  uint16_t sc_next[4], sc_next2[4];
  load_scales(0, sc_next);
  load_scales(1, sc_next2);
  if (t == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&rbar, 1);
    if (push) mbar_arrive_expect_tx(&rbar, static_cast<uint32_t>(a.cs * own * kTcN * 4));
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base)), "n"(CFG::tmem)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (a.gain) {  // the RMSNorm gain of this rank's K range, into L2 ahead of the dependency wait
    for (int i = t; i < KR / 32; i += NT) prefetch_l2(a.gain + kc0 + 32 * i);
  }
  prefetch_share(a.pf, a.pf_bytes, NT);
  // per-pass state of the two passes in flight, kept in registers (even and
  // odd passes as separate variables: an array indexed by the pass parity
  // would live in local memory, which misses the small L1 left beside the
  // shared-memory carve-out)
  float sc0[4], sc1[4];  // block scales of the even / odd pass
  int nb0 = 0, nb1 = 0;  // blocks of the even / odd pass
  uint32_t ph0 = 0u, ph1 = 0u;
  float acc[kTcN];
#pragma unroll
  for (int b = 0; b < kTcN; ++b) acc[b] = 0.f;
  bool ok = true;
  const int b_ep = t & (kTcN - 1);  // the sequence this thread's epilogue items belong to
  float ssum = 0.f;
  float* recv = reinterpret_cast<float*>(sm + CFG::recv);
  // kEpiResid: the residual of this thread's first epilogue item, loaded with
  // the activations (one round trip) instead of after the reduction
  float res0 = 0.f, res1 = 0.f;
  bool res_pre = false;
  uint32_t lane_addr = 0;
  // read out pass q: scale each block's column sums and add them up
  auto readout = [&](int q) {
    const bool odd = q & 1;
    if (!mbar_wait_bounded(&bars[odd ? 1 : 0], odd ? ph1 : ph0, a.err)) ok = false;
    if (odd) ph1 ^= 1u;
    else ph0 ^= 1u;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int nbq = odd ? nb1 : nb0;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
      if (blk >= nbq) break;
      float v[16];
      tmem_block_sum(lane_addr + blk * kTcN3, v);
      const float scale = odd ? sc1[blk] : sc0[blk];
#pragma unroll
      for (int b = 0; b < kTcN; ++b) acc[b] = fmaf(scale, v[b], acc[b]);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  };
  // reduce one tile's sums over the cluster (each CTA pushes its partials of
  // the rows another CTA owns into that CTA's shared memory) and apply the
  // epilogue; thread t handles row pairs (2m, 2m+1) of the rows this CTA owns
  // for sequence t % 16, summing the partials in rank order
  auto epilogue = [&]() {
    const int rs = recv_stride(a.cs), row0 = tile * kTcM;
    {
      const int q = ((tr / 2 + 1) * a.cs - 1) / (kTcM / 2);  // the rank that owns row tr
      const int lr = tr - pair_row0(q, a.cs);
      const uint32_t dst = mapa_u32(recv + (rank * rs + lr) * kTcN, static_cast<uint32_t>(q));
      if (push) {
        cluster_wait();
        const uint32_t qbar = mapa_u32(&rbar, static_cast<uint32_t>(q));
#pragma unroll
        for (int i = 0; i < kTcN / 4; ++i)
          st_async4(dst + 16 * i, qbar, acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < kTcN / 4; ++i)
          st_dsmem4(dst + 16 * i, acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
      }
#pragma unroll
      for (int b = 0; b < kTcN; ++b) acc[b] = 0.f;
    }
    if (push) {
      if (!mbar_wait_bounded(&rbar, 0u, a.err)) ok = false;
    } else {
      cluster_sync();
    }
    const float scl = inv_rms[b_ep];
    for (int idx = t; idx < own * (kTcN / 2); idx += NT) {
      const int lr = 2 * (idx / kTcN);
      float v0 = 0.f, v1 = 0.f;
      for (int q = 0; q < a.cs; ++q) {
        v0 += recv[(q * rs + lr) * kTcN + b_ep];
        v1 += recv[(q * rs + lr + 1) * kTcN + b_ep];
      }
      v0 *= scl;
      v1 *= scl;
      const int r0 = row0 + own0 + lr, r1 = r0 + 1;
      if (b_ep >= a.n || r0 >= a.rows) continue;
      const bool ok1 = r1 < a.rows;
      if (a.epi == kEpiSwiGLU) {
        a.Y[static_cast<size_t>(b_ep) * a.ldy + (r0 >> 1)] = silu_mul(v0, v1);
      } else {
        float* y = a.Y + static_cast<size_t>(b_ep) * a.ldy;
        if (a.epi == kEpiResid) {
          const bool pre = res_pre && idx == t;
          v0 += pre ? res0 : y[r0];
          if (ok1) v1 += pre ? res1 : y[r1];
          ssum = fmaf(v0, v0, ssum);
          if (ok1) ssum = fmaf(v1, v1, ssum);
        }
        y[r0] = v0;
        if (ok1) y[r1] = v1;
      }
    }
  };
  // wait for pass g's weights and dequantise them into A (this thread's row,
  // both sub-chunks); with one A / tensor-memory buffer the previous pass is
  // read out first
  auto load_pass = [&](int g) {
    const int k0 = kc0 + g * PK, pk = min(PK, kc0 + KR - k0);
    if (g & 1) {
      nb1 = pk / 32;
#pragma unroll
      for (int i = 0; i < 4; ++i) sc1[i] = q8 ? __half2float(__ushort_as_half(sc_next[i])) : 1.f;
    } else {
      nb0 = pk / 32;
#pragma unroll
      for (int i = 0; i < 4; ++i) sc0[i] = q8 ? __half2float(__ushort_as_half(sc_next[i])) : 1.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) sc_next[i] = sc_next2[i];
    load_scales(g + 2, sc_next2);
    // keep STAGES - 1 passes in flight ahead of this one
    if (g + STAGES - 1 < total) issue_raw(g + STAGES - 1);
    else cp_async_commit();
    cp_async_wait<STAGES - 1>();
    __syncthreads();
    if (g > 0) readout(g - 1);
    const unsigned char* raw = sm + (g % STAGES) * kRawBytes + tr * kPassBytes;
    unsigned char* A = sm + CFG::a;
    if (q8) {
      for (int ch = 0; ch < pk / 16; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4*>(raw + ((ch ^ (tr & 7)) << 4));
        uint32_t o[8];
        i8x4_to_bf16x4(w.x, o[0], o[1]);
        i8x4_to_bf16x4(w.y, o[2], o[3]);
        i8x4_to_bf16x4(w.z, o[4], o[5]);
        i8x4_to_bf16x4(w.w, o[6], o[7]);
        unsigned char* As = A + (ch >> 2) * kABytes;
        const int kk = (ch & 3) * 16;
        *reinterpret_cast<uint4*>(As + core_off16(tr, kk)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(As + core_off16(tr, kk + 8)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    } else {
      for (int ch = 0; ch < pk / 8; ++ch)
        *reinterpret_cast<uint4*>(A + core_off16(tr, ch * 8)) =
            *reinterpret_cast<const uint4*>(raw + ((ch ^ (tr & 7)) << 4));
    }
  };
  // a CTA with two passes of one tile dequantises its second pass before the
  // wait too: that pass's quants are read from raw stage 1 into registers, and
  // after a barrier its bf16 A is written over both raw stages (A's size)
  const bool pre2 = STAGES == 2 && npass == 2;
  static_assert(CFG::a >= kAPassBytes || STAGES != 2, "pass-1 A fits the raw stages");
  auto prep_pass1 = [&]() {
    const int k0 = kc0 + PK, pk = min(PK, kc0 + KR - k0);
    nb1 = pk / 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) sc1[i] = q8 ? __half2float(__ushort_as_half(sc_next[i])) : 1.f;
    cp_async_wait<0>();
    __syncthreads();
    const unsigned char* raw = sm + kRawBytes + tr * kPassBytes;
    const int nch = q8 ? pk / 16 : pk / 8;
    uint4 w[8];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
      w[ch] = ch < nch ? *reinterpret_cast<const uint4*>(raw + ((ch ^ (tr & 7)) << 4)) : make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      if (ch >= nch) break;
      if (q8) {
        uint32_t o[8];
        i8x4_to_bf16x4(w[ch].x, o[0], o[1]);
        i8x4_to_bf16x4(w[ch].y, o[2], o[3]);
        i8x4_to_bf16x4(w[ch].z, o[4], o[5]);
        i8x4_to_bf16x4(w[ch].w, o[6], o[7]);
        unsigned char* As = sm + (ch >> 2) * kABytes;
        const int kk = (ch & 3) * 16;
        *reinterpret_cast<uint4*>(As + core_off16(tr, kk)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(As + core_off16(tr, kk + 8)) = make_uint4(o[4], o[5], o[6], o[7]);
      } else {
        *reinterpret_cast<uint4*>(sm + core_off16(tr, ch * 8)) = w[ch];
      }
    }
  };
  // the first pass's weights are dequantised before the wait as well
  if (total > 0) load_pass(0);
  if (pre2) prep_pass1();
  // every rank's rbar is initialised before any partial is sent: arrive now,
  // wait just before sending (by then every rank has long arrived)
  if (push) cluster_arrive();
  pdl_wait();
  pdl_launch_dependents();
  // inputs of the previous kernel: the RMSNorm sums of squares and B for the
  // CTA's whole K range (16 batch rows x KR activations times the gain, three
  // bf16 parts per sub-chunk: rows 0-15, 16-31, 32-47 of the N = 48 operand)
  {
    // partial sums of squares, [nss][16]: thread t adds the float4 columns of
    // sequences 4 (t % 4) .. 4 (t % 4) + 3; the first four loads per thread
    // are issued before the activations' and consumed after them
    const float4* ss4 = reinterpret_cast<const float4*>(a.ss);
    const int n4 = a.gain ? a.nss * (kTcN / 4) : 0;
    float4 sv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      sv[u] = t + u * NT < n4 ? __ldcg(ss4 + t + u * NT) : make_float4(0.f, 0.f, 0.f, 0.f);
    const int nsubs = (KR + kSubK - 1) / kSubK;
    const bool parts = a.part_o != nullptr;
    if (a.epi == kEpiResid && t < own * (kTcN / 2)) {
      const int r0 = tile * kTcM + own0 + 2 * (t / kTcN);
      if (b_ep < a.n && r0 < a.rows) {
        const float* y = a.Y + static_cast<size_t>(b_ep) * a.ldy;
        res0 = __ldcg(y + r0);
        if (r0 + 1 < a.rows) res1 = __ldcg(y + r0 + 1);
        res_pre = true;
      }
    }
    const int b = (t >> 3) & (kTcN - 1), k8 = (t & 7) * 8;
    for (int s0 = 0; s0 < nsubs; s0 += 4) {  // sub-chunks s0 .. s0 + 3
      // every load of the round first (activations, gains), arithmetic after
      float4 xv[4][2], gv[4][2];
      bool vld[4];
      const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f), one4 = make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int sidx = s0 + i;
        vld[i] = sidx < nsubs && b < a.n && k8 < min(kSubK, KR - sidx * kSubK);
        if (parts) continue;
        const float4* src = reinterpret_cast<const float4*>(
            a.X + (vld[i] ? static_cast<size_t>(b) * a.ldx + kc0 + sidx * kSubK + k8 : 0));
        xv[i][0] = vld[i] ? __ldcg(src) : zero4;
        xv[i][1] = vld[i] ? __ldcg(src + 1) : zero4;
      }
      if (parts) {
        // merge the attention chunks of each element's head by log-sum-exp,
        // two chunks per round for all four sub-chunks (branch-free, so every
        // load of a round is issued before its arithmetic)
        float M[4], L[4];
        float4 o0[4], o1[4];
        size_t base[4];
        int dd[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int k = kc0 + (s0 + i) * kSubK + k8, h = k / a.hd;
          dd[i] = k - h * a.hd;
          base[i] = (static_cast<size_t>(b) * (a.K / a.hd) + h) * a.nch;
          M[i] = -INFINITY;
          L[i] = 0.f;
          o0[i] = o1[i] = zero4;
        }
        for (int c = 0; c < a.nch; c += 2) {
          const bool two = c + 1 < a.nch;
          float2 ml[4][2];
          float4 q[4][2][2];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const bool on = vld[i] && (j == 0 || two);
              const size_t e = on ? base[i] + c + j : 0;
              ml[i][j] = __ldcg(reinterpret_cast<const float2*>(a.part_ml) + e);
              const float4* po = reinterpret_cast<const float4*>(a.part_o + (on ? e * a.hd + dd[i] : 0));
              q[i][j][0] = __ldcg(po);
              q[i][j][1] = __ldcg(po + 1);
              if (!on) {  // a placeholder load: weight zero, and no NaN from unwritten memory
                ml[i][j] = make_float2(-INFINITY, 0.f);
                q[i][j][0] = q[i][j][1] = zero4;
              }
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float Mn = fmaxf(M[i], fmaxf(ml[i][0].x, ml[i][1].x));
            const float f = M[i] == -INFINITY ? 0.f : expf(M[i] - Mn);
            const float w0 = ml[i][0].x == -INFINITY ? 0.f : expf(ml[i][0].x - Mn);
            const float w1 = ml[i][1].x == -INFINITY ? 0.f : expf(ml[i][1].x - Mn);
            L[i] = fmaf(w1, ml[i][1].y, fmaf(w0, ml[i][0].y, L[i] * f));
            o0[i].x = fmaf(w1, q[i][1][0].x, fmaf(w0, q[i][0][0].x, o0[i].x * f));
            o0[i].y = fmaf(w1, q[i][1][0].y, fmaf(w0, q[i][0][0].y, o0[i].y * f));
            o0[i].z = fmaf(w1, q[i][1][0].z, fmaf(w0, q[i][0][0].z, o0[i].z * f));
            o0[i].w = fmaf(w1, q[i][1][0].w, fmaf(w0, q[i][0][0].w, o0[i].w * f));
            o1[i].x = fmaf(w1, q[i][1][1].x, fmaf(w0, q[i][0][1].x, o1[i].x * f));
            o1[i].y = fmaf(w1, q[i][1][1].y, fmaf(w0, q[i][0][1].y, o1[i].y * f));
            o1[i].z = fmaf(w1, q[i][1][1].z, fmaf(w0, q[i][0][1].z, o1[i].z * f));
            o1[i].w = fmaf(w1, q[i][1][1].w, fmaf(w0, q[i][0][1].w, o1[i].w * f));
            M[i] = Mn == -INFINITY ? M[i] : Mn;
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool nz = L[i] > 0.f;
          xv[i][0] = nz ? make_float4(o0[i].x / L[i], o0[i].y / L[i], o0[i].z / L[i], o0[i].w / L[i]) : zero4;
          xv[i][1] = nz ? make_float4(o1[i].x / L[i], o1[i].y / L[i], o1[i].z / L[i], o1[i].w / L[i]) : zero4;
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool gl = a.gain && vld[i];
        const float4* gp = reinterpret_cast<const float4*>(gl ? a.gain + kc0 + (s0 + i) * kSubK + k8 : a.gain);
        gv[i][0] = gl ? __ldg(gp) : one4;
        gv[i][1] = gl ? __ldg(gp + 1) : one4;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xv[i][0].x *= gv[i][0].x; xv[i][0].y *= gv[i][0].y; xv[i][0].z *= gv[i][0].z; xv[i][0].w *= gv[i][0].w;
        xv[i][1].x *= gv[i][1].x; xv[i][1].y *= gv[i][1].y; xv[i][1].z *= gv[i][1].z; xv[i][1].w *= gv[i][1].w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int sidx = s0 + i;
        if (sidx >= nsubs) break;
        const float x[8] = {xv[i][0].x, xv[i][0].y, xv[i][0].z, xv[i][0].w,
                            xv[i][1].x, xv[i][1].y, xv[i][1].z, xv[i][1].w};
        uint32_t p1[8], p2[8], p3[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) split3_bf16(x[e], p1[e], p2[e], p3[e]);
        unsigned char* B = sm + CFG::b + sidx * kBBytes + core_off16(b, k8);
        *reinterpret_cast<uint4*>(B) =
            make_uint4(p1[0] | (p1[1] << 16), p1[2] | (p1[3] << 16), p1[4] | (p1[5] << 16), p1[6] | (p1[7] << 16));
        *reinterpret_cast<uint4*>(B + kBPartBytes) =
            make_uint4(p2[0] | (p2[1] << 16), p2[2] | (p2[3] << 16), p2[4] | (p2[5] << 16), p2[6] | (p2[7] << 16));
        *reinterpret_cast<uint4*>(B + 2 * kBPartBytes) =
            make_uint4(p3[0] | (p3[1] << 16), p3[2] | (p3[3] << 16), p3[4] | (p3[5] << 16), p3[6] | (p3[7] << 16));
      }
    }
    for (int i = t + 4 * NT; i < n4; i += 4 * NT) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (i + u * NT >= n4) break;
        const float4 v = __ldcg(ss4 + i + u * NT);
        sv[u].x += v.x; sv[u].y += v.y; sv[u].z += v.z; sv[u].w += v.w;
      }
    }
    float s4[4] = {(sv[0].x + sv[1].x) + (sv[2].x + sv[3].x), (sv[0].y + sv[1].y) + (sv[2].y + sv[3].y),
                   (sv[0].z + sv[1].z) + (sv[2].z + sv[3].z), (sv[0].w + sv[1].w) + (sv[2].w + sv[3].w)};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s4[e] += __shfl_xor_sync(0xFFFFFFFFu, s4[e], 4);
      s4[e] += __shfl_xor_sync(0xFFFFFFFFu, s4[e], 8);
      s4[e] += __shfl_xor_sync(0xFFFFFFFFu, s4[e], 16);
    }
    if (lane < 4) {
#pragma unroll
      for (int e = 0; e < 4; ++e) wred_v[warp][4 * lane + e] = s4[e];
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (t < kTcN) {
    float ss = 0.f;
    for (int w = 0; w < NW; ++w) ss += wred_v[w][t];
    inv_rms[t] = a.gain ? rsqrtf(ss / static_cast<float>(a.K) + a.eps) : 1.f;
  }
  const uint32_t dt = tmem_base;
  lane_addr = dt + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  for (int g = 0; g < total; ++g) {
    if (g > 0) {
      if (pre2) readout(0);  // the tensor memory is free for pass 1
      else load_pass(g);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (t == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      unsigned char* A = pre2 && g == 1 ? sm : sm + CFG::a;
      const unsigned char* Bp = sm + CFG::b + (g * PK / kSubK) * kBBytes;
      mma_pass<false>(dt, kTcN3, smem_desc(A, 128, (kSubK / 8) * 128), smem_desc(Bp, 128, (kSubK / 8) * 128),
                      kBBytes, (g & 1) ? nb1 : nb0);
      mma_commit(&bars[g & 1]);
    }
  }
  if (total > 0) readout(total - 1);
  epilogue();  // every rank takes part in the cluster's reduction
  cp_async_wait<0>();
  __syncthreads();
  if (warp == 0) {  // the tensor memory is released on every path
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(dt), "n"(CFG::tmem) : "memory");
  }
  (void)ok;  // a timed-out wait has set the error word; the host reports it
  if (a.epi == kEpiResid && a.ss_out) {
    ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, 16);
    if (lane < kTcN) wred_v[warp][lane] = ssum;
    __syncthreads();
    if (t < kTcN) {
      float v = 0.f;
      for (int w = 0; w < NW; ++w) v += wred_v[w][t];
      a.ss_out[blockIdx.x * kTcN + t] = v;
    }
    return;
  }
}

// ---------------------------------------------------------------- lm_head
// One CTA per SM loops over 128-row tiles of the lm_head, 128 K (Q8_0) or
// 64 K (bf16) per pass ("Eight kernels", lm_head_argmax, as a batched
// tensor-core contraction).  The operands are f16 here: A = the int8 quants
// (exact in f16; bf16 weights are stored rounded to f16), B = x (the final
// RMSNorm output times its gain, bounded) as two f16 parts x1 + x2, which
// carry x to 2^-22 relative; N = 32.  That halves B against the three bf16
// parts of the projections and leaves room for deeper pipelines.
// Warp-specialised:
//  * warp 12 (one thread) streams whole passes of the tile-pass copy of the
//    weights (k_tile_head) into kHdStages stages with bulk copies and issues
//    each pass's MMAs into one of kHdRegions tensor-memory regions;
//  * warps 4-11, two threads per weight row: convert the row's quants of a
//    pass into one of kHdABufs A buffers;
//  * warps 0-3, one thread per row (= tensor-memory lane): read a region out
//    while the next passes are converted and multiplied, scale the block sums
//    by the row's f16 block scales, and at a tile's end write the logits and
//    fold them into running per-sequence argmax candidates.
// mbarriers hand the passes over: full[stage] (a pass's quants have landed),
// aready[buf] (an A buffer holds a pass), afree[buf] (its MMAs are done with
// it), afull[region] (the MMAs into a region are done), tfree[region] (it has
// been read out).
constexpr int kHdStages = 4;   // raw stages
constexpr int kHdABufs = 3;    // A buffers
constexpr int kHdRegions = 4;  // tensor-memory regions of kTcN * 8 = 128 columns (four blocks of N = 32)
constexpr uint32_t kHdBBytes = 2 * kBPartBytes;  // one sub-chunk of B: two f16 parts
constexpr int kHdThreads = 416;  // read-out warps 0-3, dequantising warps 4-11, issuing warp 12
struct HeadSm {
  static constexpr uint32_t b = 0;                          // B: 16 sub-chunks of 64 K
  static constexpr uint32_t a = b + 16 * kHdBBytes;         // A: kHdABufs passes
  static constexpr uint32_t raw = a + kHdABufs * kAPassBytes;  // raw quants: kHdStages passes
  static constexpr uint32_t total = raw + kHdStages * kRawBytes;
};
static_assert(HeadSm::total + 2048 <= 227 * 1024, "lm_head CTA fits");

__device__ __forceinline__ uint2 ld_weights8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// The lm_head in tile-pass order for the batched step: for every 128-row
// tile and every pass (128 K of Q8_0, 64 K of bf16) one contiguous
// kHdPassBytes block: the 128 rows' quants of the pass (128 bytes a row, its
// 16-byte chunks already in the XOR-swizzled order the dequantisation reads),
// then the 128 rows' four f16 block scales (1.0 for bf16 weights, whose
// values are stored as f16, rounded to nearest; zero rows past the end).  One
// 1-D bulk copy then brings a whole pass.
constexpr uint32_t kHdScaleOff = kRawBytes;
constexpr uint32_t kHdPassBytes = kRawBytes + kTcM * 8;
__global__ void __launch_bounds__(kTcM) k_tile_head(const uint8_t* src, size_t rb, int rows, int K, int fmt,
                                                   uint8_t* dst) {
  const bool q8 = fmt == kFmtQ8;
  const int PK = q8 ? kPassBytes : kPassBytes / 2, npass = (K + PK - 1) / PK;
  const int tile = static_cast<int>(blockIdx.x) / npass, p = static_cast<int>(blockIdx.x) - tile * npass;
  const int r = static_cast<int>(threadIdx.x), row = tile * kTcM + r;
  const int k0 = p * PK, pk = min(PK, K - k0), chunks = (q8 ? pk : 2 * pk) / 16;
  uint8_t* d = dst + static_cast<size_t>(blockIdx.x) * kHdPassBytes;
  const uint8_t* s = src + static_cast<size_t>(row < rows ? row : 0) * rb;
  for (int ch = 0; ch < 8; ++ch) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < rows && ch < chunks) v = *reinterpret_cast<const uint4*>(s + (q8 ? k0 : 2 * k0) + 16 * ch);
    if (!q8) {  // bf16 pairs -> f16 pairs
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
      for (int j = 0; j < 4; ++j) {
        const __half2 h = __floats2half2_rn(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u));
        w[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
    *reinterpret_cast<uint4*>(d + r * kPassBytes + ((ch ^ (r & 7)) << 4)) = v;
  }
  uint16_t sc[4];
  for (int i = 0; i < 4; ++i) {
    const int blk = k0 / 32 + i;
    sc[i] = 0;
    if (row < rows && i < pk / 32) sc[i] = q8 ? *reinterpret_cast<const uint16_t*>(s + K + 2 * blk) : 0x3C00u;
  }
  *reinterpret_cast<uint2*>(d + kHdScaleOff + r * 8) =
      make_uint2(sc[0] | (static_cast<uint32_t>(sc[1]) << 16), sc[2] | (static_cast<uint32_t>(sc[3]) << 16));
}

__global__ void __launch_bounds__(kHdThreads, 1) k_head16(MmArgs a) {
  constexpr int NT = kHdThreads, NW = NT / 32;
  extern __shared__ __align__(1024) unsigned char sm[];
  __shared__ __align__(8) uint64_t aready[kHdABufs], afree[kHdABufs], afull[kHdRegions], tfree[kHdRegions];
  __shared__ __align__(8) uint64_t full[kHdStages];
  __shared__ uint32_t tmem_base;
  __shared__ float inv_rms[kTcN];
  __shared__ float wred_v[NW][kTcN];
  __shared__ int wred_i[NW][kTcN];
  __shared__ float* s_logits[kTcN];
  __shared__ uint32_t s_last;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, tr = t & (kTcM - 1);
  const bool loader = t >= kTcM && t < 3 * kTcM, issuer = t == 3 * kTcM;
  const int hf = (t >> 7) - 1;  // a dequantising thread's half of its row's chunks
  const bool q8 = a.fmt == kFmtQ8;
  const int PK = q8 ? kPassBytes : kPassBytes / 2;  // K per pass
  const int npass = (a.K + PK - 1) / PK;
  const int tiles = (a.rows + kTcM - 1) / kTcM;
  const int bx = static_cast<int>(blockIdx.x), gx = static_cast<int>(gridDim.x);
  const int ntile = bx < tiles ? (tiles - 1 - bx) / gx + 1 : 0;
  const int total = ntile * npass;  // passes of this CTA
  auto pass_row0 = [&](int g) { return (bx + (g / npass) * gx) * kTcM; };
  auto pass_k0 = [&](int g) { return (g % npass) * PK; };
  // pass g's block of the tile-pass copy (a.W)
  auto pass_src = [&](int g) {
    return a.W + (static_cast<size_t>(pass_row0(g) / kTcM) * npass + g % npass) * kHdPassBytes;
  };
  // pass g's quants -> stage g % kHdStages, one bulk copy (issued by one thread)
  auto issue_pass = [&](int g) {
    if (g >= total) return;
    uint64_t* bar = &full[g % kHdStages];
    mbar_arrive_expect_tx(bar, kRawBytes);
    bulk_g2s(sm + HeadSm::raw + (g % kHdStages) * kRawBytes, pass_src(g), kRawBytes, bar);
  };
  // this thread's half of its row of pass g, converted to f16 in A buffer g % kHdABufs
  auto dequant = [&](int g) {
    const int pk = min(PK, a.K - pass_k0(g));
    const unsigned char* raw = sm + HeadSm::raw + (g % kHdStages) * kRawBytes + tr * kPassBytes;
    unsigned char* A = sm + HeadSm::a + (g % kHdABufs) * kAPassBytes;
    if (q8) {
      for (int ch = hf; ch < pk / 16; ch += 2) {
        const uint4 w = *reinterpret_cast<const uint4*>(raw + ((ch ^ (tr & 7)) << 4));
        uint32_t o[8];
        i8x4_to_f16x4(w.x, o[0], o[1]);
        i8x4_to_f16x4(w.y, o[2], o[3]);
        i8x4_to_f16x4(w.z, o[4], o[5]);
        i8x4_to_f16x4(w.w, o[6], o[7]);
        unsigned char* As = A + (ch >> 2) * kABytes;
        const int kk = (ch & 3) * 16;
        *reinterpret_cast<uint4*>(As + core_off16(tr, kk)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(As + core_off16(tr, kk + 8)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    } else {
      for (int ch = hf; ch < pk / 8; ch += 2)
        *reinterpret_cast<uint4*>(A + core_off16(tr, ch * 8)) =
            *reinterpret_cast<const uint4*>(raw + ((ch ^ (tr & 7)) << 4));
    }
  };
  // the four f16 block scales of this thread's row in pass g
  auto load_sc = [&](int g) {
    if (g >= total) return make_uint2(0u, 0u);
    return ld_weights8(pass_src(g) + kHdScaleOff + tr * 8);
  };
  if (t == 0) {
    for (int i = 0; i < kHdABufs; ++i) {
      mbar_init(&aready[i], 2 * kTcM);
      mbar_init(&afree[i], 1);
    }
    for (int i = 0; i < kHdRegions; ++i) {
      mbar_init(&afull[i], 1);
      mbar_init(&tfree[i], kTcM);
    }
    for (int i = 0; i < kHdStages; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  if (t < kTcN) s_logits[t] = t < a.n && t >= a.out0 ? a.seqs[t].logits : nullptr;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_addr(&tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // weights never depend on earlier kernels: the first stages, pass 0's
  // dequantisation and the first scales happen before the wait
  __syncthreads();  // the barriers are initialised
  uint2 sc0 = make_uint2(0u, 0u), sc1 = sc0, sc2 = sc0, sc3 = sc0;
  if (issuer) {
    for (int g = 0; g < kHdStages; ++g) issue_pass(g);
  } else if (loader) {
    if (total > 0) {
      mbar_wait_bounded(&full[0], 0u, a.err);
      dequant(0);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&aready[0]);
    }
  } else if (t < kTcM) {
    sc0 = load_sc(0);
    sc1 = load_sc(1);
    sc2 = load_sc(2);
    sc3 = load_sc(3);
  }
  pdl_wait();
  pdl_launch_dependents();
  // B for all of K: 16 batch rows x K activations times the gain, three bf16
  // parts per sub-chunk; and the RMSNorm scale of every sequence (warps 0-7)
  constexpr int RT = 2 * kTcM, RW = RT / 32;
  if (t < RT) {
    const float4* ss4 = reinterpret_cast<const float4*>(a.ss);
    const int n4 = a.gain ? a.nss * (kTcN / 4) : 0;
    float4 sv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      sv[u] = t + u * RT < n4 ? __ldcg(ss4 + t + u * RT) : make_float4(0.f, 0.f, 0.f, 0.f);
    const int nsubs = (a.K + kSubK - 1) / kSubK;
    const int b = (t >> 3) & (kTcN - 1), k8 = (t & 7) * 8, hf = t / kTcM;
    const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f), one4 = make_float4(1.f, 1.f, 1.f, 1.f);
    for (int s0 = hf; s0 < nsubs; s0 += 8) {  // sub-chunks s0, s0 + 2, s0 + 4, s0 + 6
      float4 xv[4][2], gv[4][2];
      bool vld[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int sidx = s0 + 2 * i;
        vld[i] = sidx < nsubs && b < a.n && k8 < min(kSubK, a.K - sidx * kSubK);
        const float4* src =
            reinterpret_cast<const float4*>(a.X + (vld[i] ? static_cast<size_t>(b) * a.ldx + sidx * kSubK + k8 : 0));
        xv[i][0] = vld[i] ? __ldcg(src) : zero4;
        xv[i][1] = vld[i] ? __ldcg(src + 1) : zero4;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool gl = a.gain && vld[i];
        const float4* gp = reinterpret_cast<const float4*>(gl ? a.gain + (s0 + 2 * i) * kSubK + k8 : a.gain);
        gv[i][0] = gl ? __ldg(gp) : one4;
        gv[i][1] = gl ? __ldg(gp + 1) : one4;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int sidx = s0 + 2 * i;
        if (sidx >= nsubs) break;
        const float x[8] = {xv[i][0].x * gv[i][0].x, xv[i][0].y * gv[i][0].y, xv[i][0].z * gv[i][0].z,
                            xv[i][0].w * gv[i][0].w, xv[i][1].x * gv[i][1].x, xv[i][1].y * gv[i][1].y,
                            xv[i][1].z * gv[i][1].z, xv[i][1].w * gv[i][1].w};
        uint32_t p1[8], p2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) split2_f16(x[e], p1[e], p2[e]);
        unsigned char* B = sm + HeadSm::b + sidx * kHdBBytes + core_off16(b, k8);
        *reinterpret_cast<uint4*>(B) =
            make_uint4(p1[0] | (p1[1] << 16), p1[2] | (p1[3] << 16), p1[4] | (p1[5] << 16), p1[6] | (p1[7] << 16));
        *reinterpret_cast<uint4*>(B + kBPartBytes) =
            make_uint4(p2[0] | (p2[1] << 16), p2[2] | (p2[3] << 16), p2[4] | (p2[5] << 16), p2[6] | (p2[7] << 16));
      }
    }
    for (int i = t + 4 * RT; i < n4; i += RT) {
      const float4 v = __ldcg(ss4 + i);
      sv[0].x += v.x; sv[0].y += v.y; sv[0].z += v.z; sv[0].w += v.w;
    }
    float s4[4] = {(sv[0].x + sv[1].x) + (sv[2].x + sv[3].x), (sv[0].y + sv[1].y) + (sv[2].y + sv[3].y),
                   (sv[0].z + sv[1].z) + (sv[2].z + sv[3].z), (sv[0].w + sv[1].w) + (sv[2].w + sv[3].w)};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s4[e] += __shfl_xor_sync(0xFFFFFFFFu, s4[e], 4);
      s4[e] += __shfl_xor_sync(0xFFFFFFFFu, s4[e], 8);
      s4[e] += __shfl_xor_sync(0xFFFFFFFFu, s4[e], 16);
    }
    if (lane < 4) {
#pragma unroll
      for (int e = 0; e < 4; ++e) wred_v[warp][4 * lane + e] = s4[e];
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B and A buffer 0, for the MMAs
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (t < kTcN) {
    float ss = 0.f;
    for (int w = 0; w < RW; ++w) ss += wred_v[w][t];
    inv_rms[t] = a.gain ? rsqrtf(ss / static_cast<float>(a.K) + a.eps) : 1.f;
  }
  __syncthreads();
  const uint32_t dt = tmem_base;
  if (loader) {
    for (int g = 1; g < total; ++g) {
      mbar_wait_bounded(&full[g % kHdStages], (g / kHdStages) & 1u, a.err);
      // the MMAs of pass g - kHdABufs have read this pass's A buffer
      if (g >= kHdABufs) mbar_wait_bounded(&afree[g % kHdABufs], ((g - kHdABufs) / kHdABufs) & 1u, a.err);
      dequant(g);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&aready[g % kHdABufs]);
    }
  } else if (issuer) {
    const uint64_t dA0 = smem_desc(sm + HeadSm::a, 128, (kSubK / 8) * 128);
    const uint64_t dB0 = smem_desc(sm + HeadSm::b, 128, (kSubK / 8) * 128);
    // running counters instead of divisions by the pass count: this thread
    // paces the passes.  isrc / ip: the pass issued next (kHdStages ahead) and
    // its pass within its tile; mp: the K pass multiplied; abuf / aph: its A
    // buffer and that buffer's phase
    const uint8_t* isrc = kHdStages < total ? pass_src(kHdStages) : a.W;
    int ip = kHdStages % npass, mp = 0, abuf = 0;
    uint32_t aph = 0u;
    const size_t tile_step = (static_cast<size_t>(gx) * npass - npass + 1) * kHdPassBytes;
    for (int g = 0; g < total; ++g) {
      // every row of pass g is in its A buffer, so its stage is free
      mbar_wait_bounded(&aready[abuf], aph, a.err);
      if (g + kHdStages < total) {
        uint64_t* bar = &full[g % kHdStages];  // the stage of pass g, reused by pass g + kHdStages
        mbar_arrive_expect_tx(bar, kRawBytes);
        bulk_g2s(sm + HeadSm::raw + (g % kHdStages) * kRawBytes, isrc, kRawBytes, bar);
        if (++ip == npass) {
          ip = 0;
          isrc += tile_step;
        } else {
          isrc += kHdPassBytes;
        }
      }
      // the pass's tensor-memory region has been read out (pass g - kHdRegions)
      if (g >= kHdRegions) mbar_wait_bounded(&tfree[g % kHdRegions], ((g - kHdRegions) / kHdRegions) & 1u, a.err);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int k0 = mp * PK, nb = min(PK, a.K - k0) / 32;
      mma_pass<true>(dt + (g % kHdRegions) * (4 * kHdN), kHdN, dA0 + ((abuf * kAPassBytes) >> 4),
                     dB0 + (((k0 / kSubK) * kHdBBytes) >> 4), kHdBBytes, nb);
      mma_commit(&afull[g % kHdRegions]);
      mma_commit(&afree[abuf]);
      if (++mp == npass) mp = 0;
      if (++abuf == kHdABufs) {
        abuf = 0;
        aph ^= 1u;
      }
    }
  } else if (t < kTcM) {
    float acc[kTcN], bv[kTcN];
    int bi[kTcN];
#pragma unroll
    for (int b = 0; b < kTcN; ++b) {
      acc[b] = 0.f;
      bv[b] = -INFINITY;
      bi[b] = INT_MAX;
    }
    const uint32_t lane_addr = dt + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    for (int g = 0; g < total; ++g) {
      const int h = g % kHdRegions, nb = min(PK, a.K - pass_k0(g)) / 32;
      mbar_wait_bounded(&afull[h], (g / kHdRegions) & 1u, a.err);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const float s[4] = {__half2float(__ushort_as_half(static_cast<uint16_t>(sc0.x & 0xFFFFu))),
                          __half2float(__ushort_as_half(static_cast<uint16_t>(sc0.x >> 16))),
                          __half2float(__ushort_as_half(static_cast<uint16_t>(sc0.y & 0xFFFFu))),
                          __half2float(__ushort_as_half(static_cast<uint16_t>(sc0.y >> 16)))};
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        if (blk >= nb) break;
        uint32_t r0[16], r1[16];  // the block's two parts
        tmem_ld16(lane_addr + h * (4 * kHdN) + blk * kHdN, r0);
        tmem_ld16(lane_addr + h * (4 * kHdN) + blk * kHdN + kTcN, r1);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int b = 0; b < kTcN; ++b)
          acc[b] = fmaf(s[blk], __uint_as_float(r0[b]) + __uint_as_float(r1[b]), acc[b]);
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      mbar_arrive(&tfree[h]);
      sc0 = sc1;
      sc1 = sc2;
      sc2 = sc3;
      sc3 = load_sc(g + 4);
      if (g % npass == npass - 1) {  // the tile's logits, into the running candidates
        const int row = pass_row0(g) + tr;
#pragma unroll
        for (int b = 0; b < kTcN; ++b) {
          const float val = acc[b] * inv_rms[b];
          acc[b] = 0.f;
          if (b < a.n && b >= a.out0 && row < a.rows) {
            s_logits[b][row] = val;
            argmax_merge(bv[b], bi[b], val, row);
          }
        }
      }
    }
    // this CTA's candidate per sequence
#pragma unroll
    for (int b = 0; b < kTcN; ++b) {
      warp_argmax(bv[b], bi[b]);
      if (lane == 0) {
        wred_v[warp][b] = bv[b];
        wred_i[warp][b] = bi[b];
      }
    }
    named_sync(2, kTcM);
    if (t < a.n && t >= a.out0) {
      float cv = -INFINITY;
      int ci = INT_MAX;
      for (int w = 0; w < kTcM / 32; ++w) argmax_merge(cv, ci, wred_v[w][t], wred_i[w][t]);
      a.seqs[t].amax_v[bx] = cv;
      a.seqs[t].amax_i[bx] = ci;
    }
  }
  // a timed-out wait has set the error word; the host reports it
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {  // every MMA has completed (its half was read out) and every read-out is done
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(dt) : "memory");
  }
  // the last CTA to arrive picks every sequence's winner
  if (t == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(a.count, 1u);
    s_last = old == gridDim.x - 1u;
    if (s_last) __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  for (int q = a.out0 + warp; q < a.n; q += NW) {
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
      s.state->last = next;
      s.state->pos = pos + 1;
      s.state->steps += 1;
    }
  }
  if (t == 0) *a.count = 0u;
}

// CTAs per tile (the cluster) for a [rows x K] projection.  A rank's share of
// K is whole 32-wide blocks (ceil(blocks / cs) at most), which must fit the
// CTA's B buffer.  Each 128-K pass of a CTA's share adds a dependent
// dequantise / MMA / read-out round after the activations arrive, so the
// fewest passes win.  Among those: if some sizes keep the launch at one CTA
// per SM (the next kernel's CTAs then find room to start early), the largest
// of them (the shortest last pass); otherwise the smallest size (the fewest
// CTAs) that still fits one wave at two CTAs per SM.  0 if no size fits.
int mm_cluster(int K, int rows, int num_sms) {
  const int tiles = (rows + kTcM - 1) / kTcM, nbk = K / 32;
  if (K % 32 != 0) return 0;
  int fallback = 0, best_passes = 0;
  for (int c = 1; c <= kMaxCluster && c <= nbk; ++c) {  // the fewest passes within one wave
    const int kr = 32 * ((nbk + c - 1) / c);
    if (kr > kSplitMaxK) continue;
    if (!fallback) fallback = c;
    const int passes = (kr + kPassBytes - 1) / kPassBytes;
    if (tiles * c <= 2 * num_sms && (!best_passes || passes < best_passes)) best_passes = passes;
  }
  if (!best_passes) return fallback;
  int one_per_sm = 0, smallest = 0;
  for (int c = 1; c <= kMaxCluster && c <= nbk; ++c) {
    const int kr = 32 * ((nbk + c - 1) / c);
    if (kr > kSplitMaxK || (kr + kPassBytes - 1) / kPassBytes != best_passes || tiles * c > 2 * num_sms) continue;
    if (!smallest) smallest = c;
    if (tiles * c <= num_sms) one_per_sm = c;
  }
  return one_per_sm ? one_per_sm : smallest;
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
// eight consumer warps run the online softmax and the block writes its
// chunk's partial (max, sum, weighted V) per head; the O projection merges the
// chunks by log-sum-exp while it stages its input ("Eight kernels",
// attention_decode, as a split-K flash decode).
constexpr int kAW = 8;                  // consumer warps
constexpr int kAT = kAW * 32;           // consumer threads
constexpr int kASlots = 3;
constexpr uint32_t kASlotBytes = 32 * 1024;

__device__ __forceinline__ void async() { asm volatile("bar.sync 1, %0;" ::"n"(kAT) : "memory"); }

// Four consecutive cache elements as floats: f32 rows, or f16 rows (8 bytes).
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __half* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  __half2 lo, hi;
  memcpy(&lo, &u.x, 4);
  memcpy(&hi, &u.y, 4);
  const float2 a = __half22float2(lo), b = __half22float2(hi);
  return make_float4(a.x, a.y, b.x, b.y);
}

// fresh: the step's own K/V row comes from qkv (normalised, rotated and
// appended here); otherwise every row up to the position is already in the
// cache (a prefill tile's rows, appended by k_kv_append_batch) and the
// producer waits for that kernel before copying.  KV16: the cache holds f16
// elements (the fresh row is rounded as it is stored and used rounded).
template <int HD, int G, bool KV16>
__device__ void attn_batch_item(const DevModel& m, const DevSeq& s, int layer, int g, int c, int nch,
                                const float* qkv, float* po, float* pml, unsigned char* sm, bool fresh) {
  using KT = typename std::conditional<KV16, __half, float>::type;
  constexpr uint32_t ES = sizeof(KT);
  constexpr int NJ = HD / 32;
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
  const bool has_new = fresh && t0 <= static_cast<int>(pos) && static_cast<int>(pos) < t1;
  const int tc = fresh ? min(t1, static_cast<int>(pos)) : t1;
  const int rpp = static_cast<int>(kASlotBytes / (2u * ES * HD));
  const size_t head = (static_cast<size_t>(layer) * m.nkv + g) * m.max_seq * HD;
  KT* kc = reinterpret_cast<KT*>(s.kcache);
  KT* vc = reinterpret_cast<KT*>(s.vcache);
  uint32_t* err = &s.state->err;
  if (threadIdx.x == kAT) {
    // producer
    if (!fresh) pdl_wait();  // this tile's rows are written by the previous kernel
    uint32_t n = 0;
    for (int a0 = t0; a0 < tc; a0 += rpp, ++n) {
      const int cnt = min(rpp, tc - a0);
      const uint32_t slot = n % kASlots, use = n / kASlots;
      if (use > 0 && !mbar_wait_bounded(empty + slot, (use - 1) & 1u, err)) break;
      const uint32_t bytes = static_cast<uint32_t>(cnt) * HD * ES;
      unsigned char* dst = sm + slot * kASlotBytes;
      mbar_arrive_expect_tx(full + slot, 2u * bytes);
      bulk_g2s(dst, kc + head + static_cast<size_t>(a0) * HD, bytes, full + slot);
      bulk_g2s(dst + static_cast<size_t>(rpp) * HD * ES, vc + head + static_cast<size_t>(a0) * HD, bytes,
               full + slot);
    }
    {  // the O projection's weights into L2, this CTA's share of their 128-byte lines
      const uint8_t* p = m.layers[layer].wo;
      const size_t lines = (m.row_bytes_qw * m.H) >> 7;
      for (size_t i = blockIdx.x; i < lines; i += gridDim.x) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + (i << 7)));
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
      if constexpr (KV16) {
        const __half hk = __float2half_rn(kv[j]), hv = __float2half_rn(vv[j]);
        kc[r + lane + 32 * j] = hk;
        vc[r + lane + 32 * j] = hv;
        kv[j] = __half2float(hk);
        vv[j] = __half2float(hv);
      } else {
        kc[r + lane + 32 * j] = kv[j];
        vc[r + lane + 32 * j] = vv[j];
      }
      knew[lane + 32 * j] = kv[j];
      vnew[lane + 32 * j] = vv[j];
    }
  }
  async();
  // Each warp takes four rows per step, eight lanes per row: lane (rg, g8)
  // holds elements 32i + 4 g8 + {0..3} (i < HD/32) of its row, so a group's
  // 16-byte reads are contiguous and a score needs a 3-step shuffle.  Every
  // group keeps its own online-softmax state over the rows it saw; the four
  // groups are merged at the end.
  constexpr int NC4 = HD / 32;        // float4 chunks per lane
  const int rg = lane >> 3, g8 = lane & 7;
  float4 qv[G][NC4], oo[G][NC4];
  float mm[G], ll[G];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    mm[hh] = -INFINITY;
    ll[hh] = 0.f;
#pragma unroll
    for (int i = 0; i < NC4; ++i) {
      qv[hh][i] = *reinterpret_cast<const float4*>(qs + hh * HD + 32 * i + 4 * g8);
      oo[hh][i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // one row for this lane's group (all 32 lanes call it; `valid` masks the
  // update); rows of the cache (KT) or the fresh row (f32)
  auto row_update = [&](const auto* kr, const auto* vr, bool valid) {
    float4 kf[NC4];
#pragma unroll
    for (int i = 0; i < NC4; ++i) kf[i] = ld4(kr + 32 * i + 4 * g8);
    float sc[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float d = 0.f;
#pragma unroll
      for (int i = 0; i < NC4; ++i) {
        d = fmaf(qv[hh][i].x, kf[i].x, d);
        d = fmaf(qv[hh][i].y, kf[i].y, d);
        d = fmaf(qv[hh][i].z, kf[i].z, d);
        d = fmaf(qv[hh][i].w, kf[i].w, d);
      }
      d += __shfl_xor_sync(0xFFFFFFFFu, d, 1);
      d += __shfl_xor_sync(0xFFFFFFFFu, d, 2);
      d += __shfl_xor_sync(0xFFFFFFFFu, d, 4);
      sc[hh] = d * m.attn_scale;
    }
    if (!valid) return;
    float4 vf[NC4];
#pragma unroll
    for (int i = 0; i < NC4; ++i) vf[i] = ld4(vr + 32 * i + 4 * g8);
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float corr = 1.f, p = 1.f;
      if (sc[hh] > mm[hh]) {
        corr = expf(mm[hh] - sc[hh]);
        mm[hh] = sc[hh];
      } else {
        p = expf(sc[hh] - mm[hh]);
      }
      ll[hh] = fmaf(ll[hh], corr, p);
#pragma unroll
      for (int i = 0; i < NC4; ++i) {
        oo[hh][i].x = fmaf(p, vf[i].x, oo[hh][i].x * corr);
        oo[hh][i].y = fmaf(p, vf[i].y, oo[hh][i].y * corr);
        oo[hh][i].z = fmaf(p, vf[i].z, oo[hh][i].z * corr);
        oo[hh][i].w = fmaf(p, vf[i].w, oo[hh][i].w * corr);
      }
    }
  };
  uint32_t n = 0;
  for (int a0 = t0; a0 < tc; a0 += rpp, ++n) {
    const int cnt = min(rpp, tc - a0);
    const uint32_t slot = n % kASlots;
    mbar_wait_bounded(full + slot, (n / kASlots) & 1u, err);
    const KT* Ks = reinterpret_cast<const KT*>(sm + slot * kASlotBytes);
    const KT* Vs = Ks + static_cast<size_t>(rpp) * HD;
    for (int r0 = 4 * warp; r0 < cnt; r0 += 4 * kAW) {
      const int r = min(r0 + rg, cnt - 1);
      row_update(Ks + r * HD, Vs + r * HD, r0 + rg < cnt);
    }
    __syncwarp();
    if (lane == 0)
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(empty + slot)) : "memory");
  }
  if (has_new && warp == kAW - 1) row_update(static_cast<const float*>(knew), static_cast<const float*>(vnew), rg == 0);
  // merge the four groups of the warp (lanes g8, g8+8, g8+16, g8+24 hold the
  // same elements), then publish the warp's state
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    float M = mm[hh];
    M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, 8));
    M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, 16));
    const float f = M == -INFINITY ? 0.f : expf(mm[hh] - M);
    float l = ll[hh] * f;
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 8);
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 16);
    float* w = wst + (warp * G + hh) * (HD + 2);
#pragma unroll
    for (int i = 0; i < NC4; ++i) {
      float4 o = oo[hh][i];
      o.x *= f; o.y *= f; o.z *= f; o.w *= f;
      o.x += __shfl_xor_sync(0xFFFFFFFFu, o.x, 8);
      o.y += __shfl_xor_sync(0xFFFFFFFFu, o.y, 8);
      o.z += __shfl_xor_sync(0xFFFFFFFFu, o.z, 8);
      o.w += __shfl_xor_sync(0xFFFFFFFFu, o.w, 8);
      o.x += __shfl_xor_sync(0xFFFFFFFFu, o.x, 16);
      o.y += __shfl_xor_sync(0xFFFFFFFFu, o.y, 16);
      o.z += __shfl_xor_sync(0xFFFFFFFFu, o.z, 16);
      o.w += __shfl_xor_sync(0xFFFFFFFFu, o.w, 16);
      if (rg == 0) {
        w[32 * i + 4 * g8] = o.x;
        w[32 * i + 4 * g8 + 1] = o.y;
        w[32 * i + 4 * g8 + 2] = o.z;
        w[32 * i + 4 * g8 + 3] = o.w;
      }
    }
    if (lane == 0) {
      w[HD] = M;
      w[HD + 1] = l;
    }
  }
  async();
  const int stride = HD + 2;
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
    po[(static_cast<size_t>(h) * nch + c) * HD + d] = O;
    if (d == 0) {
      pml[(static_cast<size_t>(h) * nch + c) * 2] = M;
      pml[(static_cast<size_t>(h) * nch + c) * 2 + 1] = Ls;
    }
  }
}

// A prefill tile's K/V rows: for slot b (one block) and kv head g (one warp),
// k after QK-norm and RoPE at the slot's position, and v, into the cache rows
// that the attention kernel then reads (the tile's slots attend to each
// other's rows, so they are written before any slot's attention starts).
// KV16: the rows are stored rounded to f16.
template <int HD, bool KV16>
__global__ void __launch_bounds__(1024) k_kv_append_batch(DevModel m, const DevSeq* seqs, int layer, const float* QKV) {
  constexpr int NJ = HD / 32;
  pdl_wait();  // this layer's QKV projection is complete
  pdl_launch_dependents();
  const int b = blockIdx.x, g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (g >= m.nkv) return;
  const DevSeq& s = seqs[b];
  const uint32_t pos = s.state->pos;
  if (pos >= static_cast<uint32_t>(m.max_seq)) return;  // flagged by the embedding
  const float* qkv = QKV + static_cast<size_t>(b) * (m.qw + 2 * m.kvw);
  float kv[NJ], vv[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    kv[j] = __ldcg(qkv + m.qw + g * HD + lane + 32 * j);
    vv[j] = __ldcg(qkv + m.qw + m.kvw + g * HD + lane + 32 * j);
  }
  head_norm_rope<HD>(kv, m.qk_norm ? m.layers[layer].k_norm : nullptr, m.rope + static_cast<size_t>(pos) * (HD / 2),
                     m.eps);
  const size_t r = ((static_cast<size_t>(layer) * m.nkv + g) * m.max_seq + pos) * HD;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    if constexpr (KV16) {
      reinterpret_cast<__half*>(s.kcache)[r + lane + 32 * j] = __float2half_rn(kv[j]);
      reinterpret_cast<__half*>(s.vcache)[r + lane + 32 * j] = __float2half_rn(vv[j]);
    } else {
      s.kcache[r + lane + 32 * j] = kv[j];
      s.vcache[r + lane + 32 * j] = vv[j];
    }
  }
}

template <int HD, int G, bool KV16>
__global__ void __launch_bounds__(kAT + 32, 2)
    k_attn_batch(DevModel m, const DevSeq* seqs, int layer, int nch, const float* QKV, float* PO, float* PML,
                 int fresh) {
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
  float* po = PO + static_cast<size_t>(b) * m.nq * nch * HD;
  float* pml = PML + static_cast<size_t>(b) * m.nq * nch * 2;
  attn_batch_item<HD, G, KV16>(m, s, layer, g, c, nch, qkv, po, pml, sm, fresh != 0);
}

// The attention kernel instantiated for the model's head_dim, group size and
// cache element type.
template <bool KV16>
const void* attn_batch_fn_t(int hd, int G) {
  if (hd == 128) {
    switch (G) {
      case 1: return reinterpret_cast<const void*>(&k_attn_batch<128, 1, KV16>);
      case 2: return reinterpret_cast<const void*>(&k_attn_batch<128, 2, KV16>);
      case 3: return reinterpret_cast<const void*>(&k_attn_batch<128, 3, KV16>);
      default: return reinterpret_cast<const void*>(&k_attn_batch<128, 4, KV16>);
    }
  }
  switch (G) {
    case 1: return reinterpret_cast<const void*>(&k_attn_batch<64, 1, KV16>);
    case 2: return reinterpret_cast<const void*>(&k_attn_batch<64, 2, KV16>);
    case 3: return reinterpret_cast<const void*>(&k_attn_batch<64, 3, KV16>);
    default: return reinterpret_cast<const void*>(&k_attn_batch<64, 4, KV16>);
  }
}

const void* attn_batch_fn(const DevModel& m) {
  const int G = m.nq / m.nkv;
  return m.kv16 ? attn_batch_fn_t<true>(m.hd, G) : attn_batch_fn_t<false>(m.hd, G);
}

size_t attn_batch_smem(const DevModel& m) {
  const int G = m.nq / m.nkv;
  return kASlots * kASlotBytes + 16 * kASlots +
         4u * (G * m.hd + 2 * m.hd + kAW * G * (m.hd + 2));
}

}  // namespace

int batch_max() { return kTcN; }

size_t batch_head_bytes(int rows, int K, int fmt) {
  const int PK = fmt == kFmtQ8 ? kPassBytes : kPassBytes / 2;
  return static_cast<size_t>((rows + kTcM - 1) / kTcM) * ((K + PK - 1) / PK) * kHdPassBytes;
}

cudaError_t launch_head_tile(const uint8_t* rows_src, size_t rb, int rows, int K, int fmt, uint8_t* dst,
                             cudaStream_t st) {
  const int PK = fmt == kFmtQ8 ? kPassBytes : kPassBytes / 2;
  const int blocks = ((rows + kTcM - 1) / kTcM) * ((K + PK - 1) / PK);
  k_tile_head<<<blocks, kTcM, 0, st>>>(rows_src, rb, rows, K, fmt, dst);
  return cudaGetLastError();
}

int batch_ss_slots(int H) { return ((H + kTcM - 1) / kTcM) * kMaxCluster; }

bool batch_supported(const DevModel& m) {
  const int G = m.nq / m.nkv;
  auto split_ok = [](int K) { return K % 64 == 0 && mm_cluster(K, kTcM, 1) > 0; };
  return G >= 1 && G <= 4 && m.nkv <= 32 && (m.hd == 64 || m.hd == 128) && split_ok(m.H) && split_ok(m.qw) &&
         split_ok(m.I) && m.H <= kHeadMaxK && attn_batch_smem(m) <= 227 * 1024;
}

namespace {

// Host-supplied tokens of one batched step: tok[b] becomes sequence b's input
// token at its next position (one upload for all sequences).
__global__ void k_batch_tokens_in(const DevSeq* seqs, int n, const int32_t* tok) {
  const int b = static_cast<int>(threadIdx.x);
  if (b < n) seqs[b].tokens[seqs[b].state->pos] = tok[b];
}

// After a step: out[b] = sequence b's argmax (its input token at the new
// position), out[n + b] = its error word (one readback for all sequences).
__global__ void k_batch_tokens_out(const DevSeq* seqs, int n, int32_t* out) {
  const int b = static_cast<int>(threadIdx.x);
  if (b < n) {
    const DevSeq& s = seqs[b];
    out[b] = s.tokens[s.state->pos];
    out[n + b] = static_cast<int32_t>(s.state->err);
  }
}

// A prefill tile: slot b is the sequence at position p0 + b, p0 being the
// sequence's next position.  slots[0 .. kTcN) share the sequence's tokens and
// KV cache, each with a state word of its own; slots[kTcN] is the sequence.
__global__ void k_prefill_tile_begin(const DevSeq* slots, int n) {
  const int b = static_cast<int>(threadIdx.x);
  if (b < n) slots[b].state->pos = slots[kTcN].state->pos + static_cast<uint32_t>(b);
}

// After a tile: the sequence advances by n positions and takes over the
// slots' error bits.
__global__ void k_prefill_tile_end(const DevSeq* slots, int n) {
  if (threadIdx.x != 0) return;
  DevState* seq = slots[kTcN].state;
  uint32_t err = 0u;
  for (int b = 0; b < n; ++b) {
    err |= slots[b].state->err;
    slots[b].state->err = 0u;
  }
  seq->err |= err;
  seq->pos += static_cast<uint32_t>(n);
  seq->steps += static_cast<uint32_t>(n);
}

}  // namespace

cudaError_t launch_batch_tokens_in(const DevSeq* seqs, int n, const int32_t* tok, cudaStream_t st) {
  k_batch_tokens_in<<<1, 64, 0, st>>>(seqs, n, tok);  // n <= 64 (tqd_config.max_batch)
  return cudaGetLastError();
}

cudaError_t launch_batch_tokens_out(const DevSeq* seqs, int n, int32_t* out, cudaStream_t st) {
  k_batch_tokens_out<<<1, 64, 0, st>>>(seqs, n, out);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tile_begin(const DevSeq* slots, int n, cudaStream_t st) {
  k_prefill_tile_begin<<<1, kTcN, 0, st>>>(slots, n);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tile_end(const DevSeq* slots, int n, cudaStream_t st) {
  k_prefill_tile_end<<<1, 32, 0, st>>>(slots, n);
  return cudaGetLastError();
}

cudaError_t batch_setup(const DevModel& m) {
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&k_mm16<SplitCfg>),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SplitCfg::total));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&k_mm16<SplitCfg>),
                           cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&k_head16), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(HeadSm::total));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_batch_fn(m), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(attn_batch_smem(m)));
}

// One batched step for sequences seqs[0..n): embedding, every layer, lm_head
// and argmax.  X, QKV, ATTN, H are batch activations; SS holds the partial
// sums of squares of x ([slots][16]) and of x after attention (the next
// [slots][16]).  Every kernel is launched with programmatic dependent launch:
// it starts streaming its weights (or cached K/V rows) while its predecessor
// finishes, and waits for it before touching activations.
// tile: seqs are the slots of one sequence's prefill tile (positions p0 ..
// p0 + n - 1), which attend to each other's rows: each layer's K/V rows are
// appended by their own kernel before the attention.  out0: the first slot
// whose logits and argmax are produced; out0 >= n skips the lm_head.
cudaError_t enqueue_batch_step(const DevModel& m, const DevLayer* host_layers, const uint8_t* lm_tiled,
                               const DevSeq* seqs, int n, int nch, float* X, float* QKV, float* PO, float* PML,
                               float* H, float* SS, uint32_t* count, uint32_t* err, cudaStream_t st, bool tile,
                               int out0) {
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
  cudaError_t e0;
  int dev = 0, num_sms = 0;
  if ((e0 = cudaGetDevice(&dev)) != cudaSuccess ||
      (e0 = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e0;
  float* ss_x = SS;                                       // after the embedding / down projection
  float* ss_mid = SS + batch_ss_slots(m.H) * kTcN;        // after the O projection
  const int nss_x = tiles_h * mm_cluster(m.I, m.H, num_sms), nss_mid = tiles_h * mm_cluster(m.qw, m.H, num_sms);
  cudaLaunchConfig_t ce = config(n, 256, 0, 1);
  cudaError_t e = cudaLaunchKernelEx(&ce, k_embed_batch, m, seqs, n, X, ss_x, nss_x);
  if (e != cudaSuccess) return e;
  auto mm = [&](const uint8_t* W, size_t rb, int K, int rows, const float* Xin, int ldx, const float* gain,
                const float* ss, int nss, int epi, float* Y, int ldy, float* ss_out, bool split,
                bool from_parts = false, const uint8_t* pf = nullptr, size_t pf_bytes = 0) {
    MmArgs a{};
    a.W = W; a.rb = rb; a.K = K; a.rows = rows; a.fmt = fmt;
    a.cs = split ? mm_cluster(K, rows, num_sms) : 1;
    a.X = Xin; a.ldx = ldx; a.n = n; a.gain = gain; a.ss = ss; a.nss = nss; a.eps = m.eps;
    a.epi = epi; a.Y = Y; a.ldy = ldy; a.ss_out = ss_out;
    a.seqs = seqs; a.count = count; a.err = err; a.max_seq = m.max_seq; a.out0 = out0;
    a.pf = pf;
    a.pf_bytes = pf_bytes;
    if (from_parts) {  // X is the attention's chunk partials, merged while B is built
      a.part_o = PO; a.part_ml = PML; a.nch = nch; a.hd = m.hd;
    }
    const int tiles = (rows + kTcM - 1) / kTcM;
    if (split) {
      cudaLaunchConfig_t c = config(tiles * a.cs, SplitCfg::threads, SplitCfg::total, a.cs);
      return cudaLaunchKernelEx(&c, k_mm16<SplitCfg>, a);
    }
    cudaLaunchConfig_t c = config(std::min(tiles, num_sms), kHdThreads, HeadSm::total, 1);
    return cudaLaunchKernelEx(&c, k_head16, a);
  };
  const int lqkv = m.qw + 2 * m.kvw;
  const void* attn_fn = attn_batch_fn(m);
  for (int l = 0; l < m.n_layers; ++l) {
    const DevLayer& L = host_layers[l];
    if ((e = mm(L.wqkv, m.row_bytes_h, m.H, lqkv, X, m.H, L.attn_norm, ss_x, nss_x, kEpiStore, QKV, lqkv,
                nullptr, true)) != cudaSuccess)
      return e;
    if (tile) {
      cudaLaunchConfig_t cp = config(n, 32 * m.nkv, 0, 1);
      const float* q = QKV;
      if (m.kv16)
        e = m.hd == 128 ? cudaLaunchKernelEx(&cp, k_kv_append_batch<128, true>, m, seqs, l, q)
                        : cudaLaunchKernelEx(&cp, k_kv_append_batch<64, true>, m, seqs, l, q);
      else
        e = m.hd == 128 ? cudaLaunchKernelEx(&cp, k_kv_append_batch<128, false>, m, seqs, l, q)
                        : cudaLaunchKernelEx(&cp, k_kv_append_batch<64, false>, m, seqs, l, q);
      if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t ca = config(n * m.nkv * nch, kAT + 32, attn_batch_smem(m), 1);
    {
      DevModel mm_ = m;
      const DevSeq* sq = seqs;
      int layer = l, nc = nch, fresh = tile ? 0 : 1;
      const float* q = QKV;
      float* po = PO;
      float* pml = PML;
      void* args[] = {&mm_, &sq, &layer, &nc, &q, &po, &pml, &fresh};
      if ((e = cudaLaunchKernelExC(&ca, attn_fn, args)) != cudaSuccess) return e;
    }
    if ((e = mm(L.wo, m.row_bytes_qw, m.qw, m.H, nullptr, m.qw, nullptr, nullptr, 0, kEpiResid, X, m.H, ss_mid,
                true, true, L.wgu, m.row_bytes_h * 2 * m.I)) != cudaSuccess)
      return e;
    if ((e = mm(L.wgu, m.row_bytes_h, m.H, 2 * m.I, X, m.H, L.ffn_norm, ss_mid, nss_mid, kEpiSwiGLU, H, m.I,
                nullptr, true, false, L.wd, m.row_bytes_i * m.H)) != cudaSuccess)
      return e;
    const bool more = l + 1 < m.n_layers;
    if ((e = mm(L.wd, m.row_bytes_i, m.I, m.H, H, m.I, nullptr, nullptr, 0, kEpiResid, X, m.H, ss_x, true, false,
                more ? host_layers[l + 1].wqkv : nullptr, more ? m.row_bytes_h * lqkv : 0)) != cudaSuccess)
      return e;
  }
  if (out0 >= n) return cudaSuccess;
  return mm(lm_tiled, m.row_bytes_h, m.H, m.V, X, m.H, m.out_norm, ss_x, nss_x, kEpiArgmax, nullptr, 0,
            nullptr, false);
}

}  // namespace tqd
