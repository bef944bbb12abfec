// Persistent schedule: one cooperative launch runs whole decode steps (one
// tqd_decode_step, a chain of tqd_generate steps, or a prefill), one block per
// SM.  Sixteen consumer warps compute; one producer warp streams every byte
// of weights and cached K/V the block will need — its static slice of every
// phase of every layer — through a ring of shared-memory slots with 1-D bulk
// copies (TMA), running ahead of the consumers across phase and layer
// boundaries.  Weights never depend on activations, so the HBM stream keeps
// flowing while the consumers wait at the grid barriers between dependent
// phases.  Phases and op order follow the inferno.rs blog, "IV.4: One
// command buffer per token", section "One command buffer".
//
// Synchronisation: a monotonic 64-bit arrival counter (release add, acquire
// poll) between dependent phases; mbarriers for the ring; every wait is
// bounded by %globaltimer and reports through the error word instead of
// hanging.
#pragma once

#include <climits>

#include "tqd_internal.h"
#include "tqd_phases.cuh"

namespace tqd {
namespace {

constexpr int kCW = 15;                 // consumer warps (16 warps per block with the producer:
                                        // four per SM sub-partition, up to 128 registers each)
constexpr int kCT = kCW * 32;           // consumer threads
constexpr int kThreads = kCT + 32;      // + the producer warp
constexpr uint32_t kSlotBytes = 44 * 1024;
constexpr int kSlots = 4;
constexpr int kPartFloats = 320;        // per-task partial sums of one ring piece
constexpr int kRedFloats = 64 + 2 * kPartFloats;
constexpr int kMaxGain = 4;             // norm gains held per thread (H <= 4 * kCT)
constexpr int kMaxParts = 4;            // partial sums load_norm_sum adds (the down projection's copies)
constexpr int kAccCopies = 4;           // copies of the down projection's accumulator (copy b % 4: at most 38
                                        // blocks add into an address; fewer copies to read back)
// Error bits that end every block's waits; the others (a bad token id, every
// logit NaN, capacity) are reported to the host without stopping the launch.
constexpr uint32_t kFatal = kErrGridBarrier | kErrMbarrier;

// ---------------------------------------------------------------- layout
struct PLayout {
  uint32_t ring, xraw, xin, scratch, red, bars, total;
};

__host__ __device__ inline uint32_t a16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline int imax(int a, int b) { return a > b ? a : b; }

// Elements per 16-byte weight chunk, and the padded shared-memory stride of
// one chunk's x values (chunk c of lane c % 32: conflict-free 128-bit reads).
__host__ __device__ constexpr int epc_of(int fmt) { return fmt == kFmtQ8 ? 16 : 8; }
__host__ __device__ constexpr int xstride_of(int fmt) { return fmt == kFmtQ8 ? 20 : 12; }

__host__ __device__ inline PLayout playout(const DevModel& m) {
  PLayout L;
  uint32_t off = 0;
  L.ring = off;
  off += kSlots * kSlotBytes;
  L.xraw = off;
  off += a16(4u * m.H);
  const int kmax = imax(m.H, imax(m.qw, m.I));
  L.xin = off;
  off += a16(4u * (kmax / epc_of(m.wtype)) * xstride_of(m.wtype));
  const int G = m.nq / m.nkv;
  const int attn = G * m.hd + 2 * m.hd + imax(G * m.n_chunks * (m.hd + 2), kCW * G * (m.hd + 2));
  L.scratch = off;
  off += a16(4u * imax(imax(m.qw, m.I), attn));
  L.red = off;
  off += 4u * kRedFloats;
  L.bars = off;
  off += 8u * (2 * kSlots);
  L.total = off;
  return L;
}

// ---------------------------------------------------------------- sync helpers
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory"); }

// OR of a predicate over the consumer threads (uniform result).
__device__ __forceinline__ bool csync_or(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(p)), "n"(kCT)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// mbarrier wait that gives up after kWaitLimitNs or as soon as another thread
// has reported a fatal error.
__device__ __forceinline__ bool mwait(uint64_t* bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 63u) == 0) {
      if (ld_volatile_u32(err) & kFatal) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicOr(err, kErrMbarrier);
        return false;
      }
    }
  }
  return true;
}

__device__ __forceinline__ void red_release_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier, split: every block arrives once per phase; a wait for epoch e
// returns once all blocks have arrived e times in total.
__device__ __forceinline__ void gb_arrive(DevBarrier* b) {
  csync();
  if (threadIdx.x == 0) red_release_add_u64(&b->count, 1ull);
}

// Returns false on every consumer thread if the wait failed (timeout or a
// fatal error reported elsewhere).
__device__ __forceinline__ bool gb_wait(DevBarrier* b, unsigned long long target, uint32_t* err) {
  bool fail = false;
  if (threadIdx.x == 0) {
    if (ld_acquire_u64(&b->count) < target) {
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire_u64(&b->count) < target) {
        if (ld_volatile_u32(err) & kFatal) {
          fail = true;
          break;
        }
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          atomicOr(err, kErrGridBarrier);
          fail = true;
          break;
        }
      }
    }
  }
  return !csync_or(fail);
}

__device__ __forceinline__ float silu_mul_fast(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }
// floor(a / b) for 0 <= a < 2^21 and b >= 1: (a + 1/2) / b is at least 1/(2b)
// away from an integer, far more than the error of an approximate reciprocal
// and one rounded product.
__device__ __forceinline__ int small_div(int a, int b) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(static_cast<float>(b)));
  return __float2int_rz((static_cast<float>(a) + 0.5f) * r);
}
// ---------------------------------------------------------------- f32x2
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// 16 Q8_0 quants (one 16-byte chunk) against 16 x values: sum q_j x_j.
__device__ __forceinline__ float dot16_q8(uint4 w, const float4* x) {
  const float2 bias = make_float2(-8388736.0f, -8388736.0f);
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t t = wv[k] ^ 0x80808080u;
    float2 q01 = make_float2(__uint_as_float(__byte_perm(t, 0x4B000000u, 0x7640)),
                             __uint_as_float(__byte_perm(t, 0x4B000000u, 0x7641)));
    float2 q23 = make_float2(__uint_as_float(__byte_perm(t, 0x4B000000u, 0x7642)),
                             __uint_as_float(__byte_perm(t, 0x4B000000u, 0x7643)));
    q01 = fadd2(q01, bias);
    q23 = fadd2(q23, bias);
    const float4 xv = x[k];
    a0 = ffma2(q01, make_float2(xv.x, xv.y), a0);
    a1 = ffma2(q23, make_float2(xv.z, xv.w), a1);
  }
  return (a0.x + a0.y) + (a1.x + a1.y);
}

// 8 bf16 weights (one 16-byte chunk) against 8 x values.
__device__ __forceinline__ float dot8_bf16(uint4 w, const float4* x) {
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
  const float4 x0 = x[0], x1 = x[1];
  a0 = ffma2(make_float2(bf16_lo(w.x), bf16_hi(w.x)), make_float2(x0.x, x0.y), a0);
  a1 = ffma2(make_float2(bf16_lo(w.y), bf16_hi(w.y)), make_float2(x0.z, x0.w), a1);
  a0 = ffma2(make_float2(bf16_lo(w.z), bf16_hi(w.z)), make_float2(x1.x, x1.y), a0);
  a1 = ffma2(make_float2(bf16_lo(w.w), bf16_hi(w.w)), make_float2(x1.z, x1.w), a1);
  return (a0.x + a0.y) + (a1.x + a1.y);
}

// ---------------------------------------------------------------- the ring
struct Ring {
  uint8_t* base;
  uint64_t* full;
  uint64_t* empty;
  uint32_t n;  // pieces issued (producer) or consumed (consumers)
};

__device__ __forceinline__ uint8_t* slot_ptr(const Ring& r) {
  return r.base + (r.n % kSlots) * kSlotBytes;
}

// Rows of a matrix a block owns in a phase: units of `align` rows split evenly.
__device__ __forceinline__ void block_rows(int rows, int align, int b, int nb, int& r0, int& r1) {
  const int units = rows / align;
  r0 = static_cast<int>(static_cast<long long>(units) * b / nb) * align;
  r1 = static_cast<int>(static_cast<long long>(units) * (b + 1) / nb) * align;
}

// Rows per ring piece: a multiple of 2 * kCW rows (one pair per consumer
// warp) when that fits a slot, else the largest even count; at most 240.
__device__ __forceinline__ int rows_per_piece(size_t rb) {
  int r = static_cast<int>(kSlotBytes / static_cast<uint32_t>(rb));  // rows are far below 4 GB
  if (r > 240) r = 240;
  if (r >= 2 * kCW) return r / (2 * kCW) * (2 * kCW);
  return r & ~1;
}

// Rows per ring piece taking every row a slot holds (even, at most 2 kCW
// pairs' worth: two pairs per warp at most).
__device__ __forceinline__ int rows_per_piece_all(size_t rb) {
  int r = static_cast<int>(kSlotBytes / static_cast<uint32_t>(rb));
  if (r > 4 * kCW) r = 4 * kCW;
  return r & ~1;
}

// K/V rows per attention piece (K rows then V rows in one slot).
__device__ __forceinline__ int kv_rows_per_piece(int hd, int esz) {
  return static_cast<int>(kSlotBytes / (2u * esz * hd));
}

// The chunk [t0, t1) of positions item chunk c covers when S rows are live.
__device__ __forceinline__ void chunk_range(int S, int n_chunks, int c, int& t0, int& t1) {
  const int cs = (S + n_chunks - 1) / n_chunks;
  t0 = min(S, c * cs);
  t1 = min(S, t0 + cs);
}

// ---------------------------------------------------------------- work plan
// What block b does in every layer; producer and consumers derive the same
// plan.  The blocks are split into one group per kv head (blocks beyond
// n_kv_heads * (blocks / n_kv_heads) belong to none).  A group computes the
// Q, K and V rows of its head group, runs its attention chunks, combines them,
// and applies its columns of the O projection (a split over heads: the O
// product is a sum over the groups' column slices), all synchronised inside
// the group only.  Gate/up, down and the lm_head are split over all blocks.
struct Plan {
  int grp, j, bpg;   // group (-1: none), index in the group, blocks per group
  int qr0[3], qr1[3];  // QKV matrix rows: the group's q, k and v rows this block owns
  int chunk;         // attention chunk of item (grp, chunk), or -1
  int o0, o1;        // rows of the group's O column slice
  int g0, g1, v0, v1;  // gate/up rows (pairs: SwiGLU outputs g0/2 .. g1/2), lm_head rows
  int zo0, zo1, zx0, zx1;  // this block's shares of the O products (H) and of the accumulator copies
};

__device__ __forceinline__ Plan make_plan(const DevModel& m, int b, int nb) {
  Plan p;
  p.bpg = nb / m.nkv;
  p.grp = (p.bpg > 0 && b < p.bpg * m.nkv) ? b / p.bpg : -1;
  p.j = p.grp >= 0 ? b - p.grp * p.bpg : 0;
  const int G = m.nq / m.nkv, gh = G * m.hd;
  p.o0 = p.o1 = 0;
#pragma unroll
  for (int i = 0; i < 3; ++i) p.qr0[i] = p.qr1[i] = 0;
  if (p.grp >= 0) {
    block_rows(m.H, 1, p.j, p.bpg, p.o0, p.o1);
    // the group's q (gh rows), k (hd) and v (hd) rows of the QKV matrix
    const int segr[3] = {gh, m.hd, m.hd};
    const int phys[3] = {p.grp * gh, m.qw + p.grp * m.hd, m.qw + m.kvw + p.grp * m.hd};
    if (p.bpg >= 3) {
      // every block takes rows of one segment: blocks go one at a time to the
      // segment with the most rows per block (ties: the first)
      int nbk[3] = {1, 1, 1};
      for (int k = 3; k < p.bpg; ++k) {
        int best = 0;
        for (int i = 1; i < 3; ++i)
          if ((segr[i] + nbk[i] - 1) / nbk[i] > (segr[best] + nbk[best] - 1) / nbk[best]) best = i;
        ++nbk[best];
      }
      int i = 0, jj = p.j;
      while (jj >= nbk[i]) jj -= nbk[i++];
      int a, e;
      block_rows(segr[i], 1, jj, nbk[i], a, e);
      p.qr0[i] = phys[i] + a;
      p.qr1[i] = phys[i] + e;
    } else {
      // fewer than three blocks: contiguous shares of the q, k, v sequence
      int l0, l1;
      block_rows(gh + 2 * m.hd, 1, p.j, p.bpg, l0, l1);
      const int seg0[3] = {0, gh, gh + m.hd};
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int a = max(l0, seg0[i]), e = min(l1, seg0[i] + segr[i]);
        if (a < e) {
          p.qr0[i] = phys[i] + (a - seg0[i]);
          p.qr1[i] = phys[i] + (e - seg0[i]);
        }
      }
    }
  }
  p.chunk = (p.grp >= 0 && p.j < m.n_chunks) ? p.j : -1;
  block_rows(2 * m.I, 2, b, nb, p.g0, p.g1);
  block_rows(m.V, 1, b, nb, p.v0, p.v1);
  block_rows(m.H, 1, b, nb, p.zo0, p.zo1);
  block_rows(kAccCopies * m.H, 1, b, nb, p.zx0, p.zx1);
  return p;
}

// ---------------------------------------------------------------- producer
struct Producer {
  Ring r;
  uint32_t* err;
  bool ok;
  uint64_t policy;  // L2 evict-first: every byte streamed here is read once per step

  __device__ bool acquire() {
    const uint32_t slot = r.n % kSlots, use = r.n / kSlots;
    if (use > 0 && !mwait(r.empty + slot, (use - 1) & 1u, err)) ok = false;
    return ok;
  }
  __device__ void rows(const uint8_t* W, size_t rb, int r0, int r1, int rpp) {
    for (int a = r0; a < r1 && ok; a += rpp) {
      const int n = min(rpp, r1 - a);
      if (!acquire()) return;
      const uint32_t bytes = static_cast<uint32_t>(n * rb);
      uint64_t* fb = r.full + r.n % kSlots;
      mbar_arrive_expect_tx(fb, bytes);
      bulk_g2s_hint(slot_ptr(r), W + static_cast<size_t>(a) * rb, bytes, fb, policy);
      ++r.n;
    }
  }
  // K and V rows [t0, t1) of one kv head's cache (esz bytes per element: 4,
  // or 2 for an f16 cache): K rows then V rows in one slot.
  __device__ void kv(const uint8_t* kc, const uint8_t* vc, int hd, int esz, int t0, int t1) {
    const int rpp = kv_rows_per_piece(hd, esz);
    const size_t rb = static_cast<size_t>(hd) * esz;
    for (int a = t0; a < t1 && ok; a += rpp) {
      const int n = min(rpp, t1 - a);
      if (!acquire()) return;
      const uint32_t bytes = static_cast<uint32_t>(n * rb);
      uint64_t* fb = r.full + r.n % kSlots;
      uint8_t* dst = slot_ptr(r);
      mbar_arrive_expect_tx(fb, 2u * bytes);
      bulk_g2s_hint(dst, kc + a * rb, bytes, fb, policy);
      bulk_g2s_hint(dst + rpp * rb, vc + a * rb, bytes, fb, policy);
      ++r.n;
    }
  }

  // Columns [j0, j1) of the down projection in its column-block layout
  // (DevModel::dcol_bytes).  Q8_0: one piece per 32-column block touched, the
  // block's scales then the quant runs of those columns; bf16: whole columns,
  // as many as a slot holds.
  __device__ void dcols(const uint8_t* Wc, const DevModel& m, int j0, int j1) {
    if (m.wtype == kFmtQ8) {
      const uint32_t sb = a16(2u * m.H);
      for (int c = j0 / 32; c * 32 < j1 && ok; ++c) {
        const int ja = max(j0, 32 * c), jb = min(j1, 32 * c + 32);
        if (!acquire()) return;
        const uint8_t* blk = Wc + static_cast<size_t>(c) * m.dcol_bytes;
        const uint32_t qb = static_cast<uint32_t>(jb - ja) * m.H;
        uint64_t* fb = r.full + r.n % kSlots;
        uint8_t* dst = slot_ptr(r);
        mbar_arrive_expect_tx(fb, sb + qb);
        bulk_g2s_hint(dst, blk, sb, fb, policy);
        bulk_g2s_hint(dst + sb, blk + sb + static_cast<size_t>(ja - 32 * c) * m.H, qb, fb, policy);
        ++r.n;
      }
    } else {
      const int cpp = static_cast<int>(kSlotBytes / (2u * m.H));
      for (int a = j0; a < j1 && ok; a += cpp) {
        const int n = min(cpp, j1 - a);
        if (!acquire()) return;
        const uint32_t bytes = static_cast<uint32_t>(n) * 2u * m.H;
        uint64_t* fb = r.full + r.n % kSlots;
        mbar_arrive_expect_tx(fb, bytes);
        bulk_g2s_hint(slot_ptr(r), Wc + static_cast<size_t>(a) * m.dcol_bytes, bytes, fb, policy);
        ++r.n;
      }
    }
  }
  // Wait until every issued copy has landed (used when stopping early).
  __device__ void drain() {
    for (uint32_t k = 0; k < kSlots && k < r.n; ++k) {
      const uint32_t q = r.n - 1 - k;
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(r.full + q % kSlots, (q / kSlots) & 1u))
        if (global_timer_ns() - t0 > kWaitLimitNs) break;
    }
  }
};

__device__ void run_producer(const DevModel& m, const DevSeq& s, int n_steps, int full_from,
                             uint32_t pos0, Ring ring) {
  Producer P{ring, &s.state->err, true, l2_evict_first_policy()};
  const Plan pl = make_plan(m, blockIdx.x, gridDim.x);
  for (int step = 0; step < n_steps && P.ok; ++step) {
    const int pos = static_cast<int>(pos0) + step;
    if (pos >= m.max_seq) break;
    for (int l = 0; l < m.n_layers && P.ok; ++l) {
      const DevLayer& L = m.layers[l];
      for (int i = 0; i < 3; ++i) P.rows(L.wqkv, m.row_bytes_h, pl.qr0[i], pl.qr1[i], rows_per_piece(m.row_bytes_h));
      if (pl.chunk >= 0) {
        int t0, t1;
        chunk_range(pos + 1, m.n_chunks, pl.chunk, t0, t1);
        const size_t head = (static_cast<size_t>(l) * m.nkv + pl.grp) * m.max_seq * m.hd;
        const int esz = m.kv16 ? 2 : 4;
        P.kv(reinterpret_cast<const uint8_t*>(s.kcache) + head * esz,
             reinterpret_cast<const uint8_t*>(s.vcache) + head * esz, m.hd, esz, t0, min(t1, pos));
      }
      if (pl.grp >= 0)
        P.rows(L.wo_g + static_cast<size_t>(pl.grp) * m.H * m.row_bytes_gh, m.row_bytes_gh, pl.o0, pl.o1,
               rows_per_piece(m.row_bytes_gh));
      P.rows(L.wgu, m.row_bytes_h, pl.g0, pl.g1, rows_per_piece_all(m.row_bytes_h));
      P.dcols(L.wd_c, m, pl.g0 / 2, pl.g1 / 2);
    }
    if (step >= full_from) P.rows(m.lm_head, m.row_bytes_h, pl.v0, pl.v1, rows_per_piece(m.row_bytes_h));
  }
  if (!P.ok) P.drain();
}

// ---------------------------------------------------------------- consumers
struct Cons {
  const DevModel& m;
  const DevSeq& s;
  Ring r;
  float* xraw;     // [H] plain vector (residual input of the phase)
  float* xin;      // matvec input in the padded chunk layout
  float* scr;      // staging / attention scratch
  float* red;      // reductions and per-task partial sums
  uint32_t rsel;   // alternating halves of the reduction scratch
  uint32_t psel;   // alternating partial-sum buffers of mv_phase
  uint32_t* err;
  int fmt;
  float inv_h;     // 1 / H (every norm of the consumers is over H values)
  __device__ Cons(const DevModel& m_, const DevSeq& s_) : m(m_), s(s_) {}
};

__device__ __forceinline__ int xpad(int fmt, int e) {
  return fmt == kFmtQ8 ? 20 * (e >> 4) + (e & 15) : 12 * (e >> 3) + (e & 7);
}

// Norm gains a thread needs, loaded before the barrier wait (they are
// constants, so their latency stays off the critical path).
struct Gain {
  float v[kMaxGain];
};
__device__ __forceinline__ void load_gain(Gain& g, const float* src, int K) {
#pragma unroll
  for (int j = 0; j < kMaxGain; ++j) {
    const int i = threadIdx.x + kCT * j;
    g.v[j] = i < K ? __ldg(src + i) : 0.f;
  }
}

// RMSNorm folded into the following matvec ("Eight kernels", rms_norm_row):
// xin <- padded(src (.) g), and the returned factor 1/sqrt(mean(src^2) + eps)
// scales every dot product, since W (x/rms (.) g) = (W (x (.) g)) / rms.
__device__ __forceinline__ float to_xin_norm(Cons& C, const float* src, int K, const Gain& g) {
  float* red = C.red + 16 * C.rsel;
  C.rsel ^= 1u;
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxGain; ++j) {
    const int i = threadIdx.x + kCT * j;
    if (i < K) {
      const float v = src[i];
      ss = fmaf(v, v, ss);
      C.xin[xpad(C.fmt, i)] = v * g.v[j];
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  csync();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kCW; ++w) t += red[w];
  return rsqrtf(fmaf(t, C.inv_h, C.m.eps));
}

// RMSNorm of a sum read from global memory (written by other blocks before
// the last grid barrier), folded into the following matvec as to_xin_norm
// does: the plain vector in xraw (the layer's input x, or x after the
// attention block) plus nparts partial sums ([nparts][K] in global memory:
// the per-group O products, or the copies of the down projection's sums),
// added in part order; xraw becomes the sum.
__device__ __forceinline__ float load_norm_sum(Cons& C, const float* parts, int nparts, int K, const Gain& g) {
  float* red = C.red + 16 * C.rsel;
  C.rsel ^= 1u;
  float v[kMaxGain];
#pragma unroll
  for (int j = 0; j < kMaxGain; ++j) {
    const int i = threadIdx.x + kCT * j;
    v[j] = i < K ? C.xraw[i] : 0.f;
  }
  // every partial is requested before any is added (one L2 round trip)
  float pv[kMaxParts][kMaxGain];
#pragma unroll
  for (int q = 0; q < kMaxParts; ++q)
#pragma unroll
    for (int j = 0; j < kMaxGain; ++j) {
      const int i = threadIdx.x + kCT * j;
      pv[q][j] = (q < nparts && i < K) ? __ldcg(parts + static_cast<size_t>(q) * K + i) : 0.f;
    }
#pragma unroll
  for (int q = 0; q < kMaxParts; ++q)
#pragma unroll
    for (int j = 0; j < kMaxGain; ++j) v[j] += pv[q][j];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxGain; ++j) {
    const int i = threadIdx.x + kCT * j;
    if (i < K) {
      ss = fmaf(v[j], v[j], ss);
      C.xraw[i] = v[j];
      C.xin[xpad(C.fmt, i)] = v[j] * g.v[j];
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  csync();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kCW; ++w) t += red[w];
  return rsqrtf(fmaf(t, C.inv_h, C.m.eps));
}

struct MvOut {
  float* y;           // kEpiStore / kEpiArgmax: y[r]; kEpiSwiGLU: y[r/2]; kEpiResid: y[r]
  const float* res;   // kEpiResid: residual source (shared memory), indexed by r
  float scale;        // multiplies every dot product (1, or 1/rms of a folded RMSNorm)
  float bv;           // running argmax (kEpiArgmax), per epilogue lane / thread
  int bi;
  uint64_t* ytag;     // kEpiTagged: ytag[r] = tag << 32 | bits of the value
  uint32_t tag;
};

// A 64-bit word written and read whole: a reader that sees the expected tag
// holds the value written with it, with no fence or counter between them.
__device__ __forceinline__ void st_tagged(uint64_t* p, uint32_t tag, float v) {
  const unsigned long long w = (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long ld_tagged(const uint64_t* p) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}

// Apply epilogue EPI to row `row` with dot product v (already scaled).
template <int EPI>
__device__ __forceinline__ void epi_row(MvOut& o, int row, float v) {
  if constexpr (EPI == kEpiTagged) {
    st_tagged(o.ytag + row, o.tag, v);
  } else if constexpr (EPI == kEpiAtomicAdd) {
    atomicAdd(o.y + row, v);
  } else if constexpr (EPI == kEpiResid) {
    o.y[row] = o.res[row] + v;
  } else {
    o.y[row] = v;
    if constexpr (EPI == kEpiArgmax) argmax_merge(o.bv, o.bi, v, row);
  }
}

// Partial dot products of rows wa and wb over chunk rounds [i0, i1) of this
// lane (chunk c = lane + 32 i), two rounds at a time for more independent
// work in flight.
template <int FMT>
__device__ __forceinline__ void dot_rows(const float* xin, const uint8_t* wa, const uint8_t* wb,
                                         int K, int nchunks, int i0, int i1, float& acc_a,
                                         float& acc_b) {
  constexpr int XS = FMT == kFmtQ8 ? 20 : 12;
  const int lane = threadIdx.x & 31;
  float a2 = 0.f, b2 = 0.f;
  int i = i0;
#pragma unroll 1
  for (; i + 1 < i1; i += 2) {
    const int c0 = lane + 32 * i, c1 = c0 + 32;
    const bool ok1 = c1 < nchunks;  // c0 < nchunks whenever c1 is
    if (c0 < nchunks) {
      const int cc1 = ok1 ? c1 : c0;
      const float4* x0 = reinterpret_cast<const float4*>(xin + XS * c0);
      const float4* x1 = reinterpret_cast<const float4*>(xin + XS * cc1);
      const uint4 wa0 = *reinterpret_cast<const uint4*>(wa + 16 * c0);
      const uint4 wb0 = *reinterpret_cast<const uint4*>(wb + 16 * c0);
      const uint4 wa1 = *reinterpret_cast<const uint4*>(wa + 16 * cc1);
      const uint4 wb1 = *reinterpret_cast<const uint4*>(wb + 16 * cc1);
      if (FMT == kFmtQ8) {
        const float sa0 = __half2float(*reinterpret_cast<const __half*>(wa + K + 2 * (c0 >> 1)));
        const float sb0 = __half2float(*reinterpret_cast<const __half*>(wb + K + 2 * (c0 >> 1)));
        const float sa1 = __half2float(*reinterpret_cast<const __half*>(wa + K + 2 * (cc1 >> 1)));
        const float sb1 = __half2float(*reinterpret_cast<const __half*>(wb + K + 2 * (cc1 >> 1)));
        const float da0 = dot16_q8(wa0, x0), db0 = dot16_q8(wb0, x0);
        const float da1 = dot16_q8(wa1, x1), db1 = dot16_q8(wb1, x1);
        acc_a = fmaf(sa0, da0, acc_a);
        acc_b = fmaf(sb0, db0, acc_b);
        if (ok1) {
          a2 = fmaf(sa1, da1, a2);
          b2 = fmaf(sb1, db1, b2);
        }
      } else {
        acc_a += dot8_bf16(wa0, x0);
        acc_b += dot8_bf16(wb0, x0);
        if (ok1) {
          a2 += dot8_bf16(wa1, x1);
          b2 += dot8_bf16(wb1, x1);
        }
      }
    }
  }
  if (i < i1) {
    const int c = lane + 32 * i;
    if (c < nchunks) {
      const float4* xp = reinterpret_cast<const float4*>(xin + XS * c);
      const uint4 w0 = *reinterpret_cast<const uint4*>(wa + 16 * c);
      const uint4 w1 = *reinterpret_cast<const uint4*>(wb + 16 * c);
      if (FMT == kFmtQ8) {
        const float s0 = __half2float(*reinterpret_cast<const __half*>(wa + K + 2 * (c >> 1)));
        const float s1 = __half2float(*reinterpret_cast<const __half*>(wb + K + 2 * (c >> 1)));
        acc_a = fmaf(s0, dot16_q8(w0, xp), acc_a);
        acc_b = fmaf(s1, dot16_q8(w1, xp), acc_b);
      } else {
        acc_a += dot8_bf16(w0, xp);
        acc_b += dot8_bf16(w1, xp);
      }
    }
  }
  acc_a += a2;
  acc_b += b2;
}

// dot_rows for two row pairs at once (rows w[0..3]), every chunk round's x
// loaded once for the four rows.
template <int FMT>
__device__ __forceinline__ void dot_rows4(const float* xin, const uint8_t* const (&w)[4], int K, int nchunks,
                                          int iters, float (&acc)[4]) {
  constexpr int XS = FMT == kFmtQ8 ? 20 : 12;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < 4; ++r) acc[r] = 0.f;
#pragma unroll 1
  for (int i = 0; i < iters; ++i) {
    const int c = lane + 32 * i;
    if (c < nchunks) {
      const float4* xp = reinterpret_cast<const float4*>(xin + XS * c);
      uint4 wv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) wv[r] = *reinterpret_cast<const uint4*>(w[r] + 16 * c);
      if (FMT == kFmtQ8) {
        float sc[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) sc[r] = __half2float(*reinterpret_cast<const __half*>(w[r] + K + 2 * (c >> 1)));
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] = fmaf(sc[r], dot16_q8(wv[r], xp), acc[r]);
      } else {
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] += dot8_bf16(wv[r], xp);
      }
    }
  }
}

// One phase of matvec rows [r0, r1) streamed through the ring, with epilogue
// EPI.  The row pairs of a piece go whole to the warps, kCW at a time (each
// warp applies the epilogue of its own pairs); the pairs left over are split
// into (pair, K segment) tasks whose partial sums go through shared memory,
// and one thread per row applies their epilogue after a consumer sync.  SHORT (rows of at most 16 chunks, K known at compile time at
// the call site) gives each half-warp its own row pair; the general path
// handles any K, short rows included.  One instance holds one path and one
// epilogue only, which keeps the per-layer code small.  WHOLE (pieces of at
// most 2 kCW pairs) takes every pair whole: a warp with two pairs computes
// both in one pass over K (four independent dot chains sharing the x loads),
// so the piece needs no K split and no consumer sync.
template <int FMT, int EPI, bool SHORT, bool WHOLE = false>
__device__ void mv_phase(Cons& C, size_t rb, int rpp, int K, int r0, int r1, MvOut& o) {
  constexpr int EPC = FMT == kFmtQ8 ? 16 : 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nchunks = K / EPC;
  const int iters = (nchunks + 31) / 32;  // chunk rounds per lane
  for (int a = r0; a < r1; a += rpp) {
    const int n = min(rpp, r1 - a);
    const int pairs = (n + 1) >> 1;
    // whole pairs kCW at a time; the pairs left over are split over K
    int full = pairs / kCW * kCW, rem = pairs - full;
    int nseg = rem > 0 ? small_div(kCW, rem) : 1;
    if (nseg > iters) nseg = iters;
    if (WHOLE || nseg <= 1) {
      nseg = 1;
      full = pairs;
      rem = 0;
    }
    const int tasks = rem * nseg;  // split tasks
    uint64_t* fb = C.r.full + C.r.n % kSlots;
    const uint8_t* slot = slot_ptr(C.r);
    float* part = C.red + 64 + kPartFloats * C.psel;  // [tasks][2] when nseg > 1
    if (nseg > 1) C.psel ^= 1u;
    // every warp waits for the piece before releasing it, so no warp can run
    // ahead and release a later use of the same slot early
    mwait(fb, (C.r.n / kSlots) & 1u, C.err);
    if constexpr (SHORT) {
      // short rows (one 16-byte chunk per lane or fewer): each half-warp takes
      // its own row pair; both halves run every round so the shuffles stay
      // warp-uniform, an idle half repeats the last pair and skips the epilogue
      constexpr int XS = FMT == kFmtQ8 ? 20 : 12;
      const int half = lane >> 4, l16 = lane & 15;
      for (int t0 = 2 * warp; t0 < pairs; t0 += 2 * kCW) {
        const int pr = min(t0 + half, pairs - 1);
        const int ra = 2 * pr, rbw = 2 * pr + 1;
        const bool has_b = rbw < n;
        const uint8_t* wa = slot + static_cast<size_t>(ra) * rb;
        const uint8_t* wb = slot + static_cast<size_t>(has_b ? rbw : ra) * rb;
        float acc_a = 0.f, acc_b = 0.f;
        if (l16 < nchunks) {
          const float4* xp = reinterpret_cast<const float4*>(C.xin + XS * l16);
          const uint4 w0 = *reinterpret_cast<const uint4*>(wa + 16 * l16);
          const uint4 w1 = *reinterpret_cast<const uint4*>(wb + 16 * l16);
          if (FMT == kFmtQ8) {
            const float s0 = __half2float(*reinterpret_cast<const __half*>(wa + K + 2 * (l16 >> 1)));
            const float s1 = __half2float(*reinterpret_cast<const __half*>(wb + K + 2 * (l16 >> 1)));
            acc_a = s0 * dot16_q8(w0, xp);
            acc_b = s1 * dot16_q8(w1, xp);
          } else {
            acc_a = dot8_bf16(w0, xp);
            acc_b = dot8_bf16(w1, xp);
          }
        }
#pragma unroll
        for (int sh = 8; sh > 0; sh >>= 1) {
          acc_a += __shfl_xor_sync(0xFFFFFFFFu, acc_a, sh);
          acc_b += __shfl_xor_sync(0xFFFFFFFFu, acc_b, sh);
        }
        if (t0 + half < pairs && l16 == 0) {
          acc_a *= o.scale;
          acc_b *= o.scale;
          if constexpr (EPI == kEpiSwiGLU) {
            o.y[(a + ra) >> 1] = silu_mul_fast(acc_a, acc_b);
          } else {
            epi_row<EPI>(o, a + ra, acc_a);
            if (has_b) epi_row<EPI>(o, a + rbw, acc_b);
          }
        }
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(C.r.empty + C.r.n % kSlots)) : "memory");
      ++C.r.n;
      continue;
    }
    if constexpr (WHOLE) {
      // at most two pairs per warp (pairs <= 2 kCW): pair warp and warp + kCW together
      const int pA = warp, pB = warp + kCW;
      if (pB < full) {
        const uint8_t* w[4];
        const int rows[4] = {2 * pA, 2 * pA + 1, 2 * pB, 2 * pB + 1};
#pragma unroll
        for (int r = 0; r < 4; ++r) w[r] = slot + static_cast<size_t>(rows[r] < n ? rows[r] : rows[r] - 1) * rb;
        float acc[4];
        dot_rows4<FMT>(C.xin, w, K, nchunks, iters, acc);
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] = warp_sum(acc[r]) * o.scale;
        if (lane == 0) {
          if constexpr (EPI == kEpiSwiGLU) {
            o.y[(a + rows[0]) >> 1] = silu_mul_fast(acc[0], acc[1]);
            o.y[(a + rows[2]) >> 1] = silu_mul_fast(acc[2], acc[3]);
          } else {
#pragma unroll
            for (int r = 0; r < 4; ++r)
              if (rows[r] < n) epi_row<EPI>(o, a + rows[r], acc[r]);
          }
        }
        full = 0;  // this warp's pairs are done
      } else if (pA >= full) {
        full = 0;
      } else {
        full = pA + 1;  // one pair: the loop below takes pair pA only
      }
    }
    for (int p = warp; p < full; p += kCW) {  // whole pairs: the warp applies the epilogue
      const int ra = 2 * p, rbw = 2 * p + 1;
      const bool has_b = rbw < n;
      float acc_a = 0.f, acc_b = 0.f;
      dot_rows<FMT>(C.xin, slot + static_cast<size_t>(ra) * rb,
                    slot + static_cast<size_t>(has_b ? rbw : ra) * rb, K, nchunks, 0, iters, acc_a, acc_b);
      acc_a = warp_sum(acc_a);
      acc_b = warp_sum(acc_b);
      if (lane == 0) {
        acc_a *= o.scale;
        acc_b *= o.scale;
        if constexpr (EPI == kEpiSwiGLU) {
          o.y[(a + ra) >> 1] = silu_mul_fast(acc_a, acc_b);
        } else {
          epi_row<EPI>(o, a + ra, acc_a);
          if (has_b) epi_row<EPI>(o, a + rbw, acc_b);
        }
      }
    }
    for (int t = warp; t < tasks; t += kCW) {  // (left-over pair, K segment): partial sums
      const int q = small_div(t, nseg), sg = t - q * nseg;
      const int ra = 2 * (full + q), rbw = ra + 1;
      const bool has_b = rbw < n;
      float acc_a = 0.f, acc_b = 0.f;
      dot_rows<FMT>(C.xin, slot + static_cast<size_t>(ra) * rb,
                    slot + static_cast<size_t>(has_b ? rbw : ra) * rb, K, nchunks,
                    small_div(iters * sg, nseg), small_div(iters * (sg + 1), nseg), acc_a, acc_b);
      acc_a = warp_sum(acc_a);
      acc_b = warp_sum(acc_b);
      if (lane == 0) {
        part[2 * t] = acc_a;
        part[2 * t + 1] = acc_b;
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(C.r.empty + C.r.n % kSlots)) : "memory");
    ++C.r.n;
    if (tasks == 0) continue;
    csync();
    // split-K epilogue of the left-over pairs: one thread per row (SwiGLU: one per pair)
    if constexpr (EPI == kEpiSwiGLU) {
      for (int q = threadIdx.x; q < rem; q += kCT) {
        float g = 0.f, u = 0.f;
        for (int sg = 0; sg < nseg; ++sg) {
          g += part[2 * (q * nseg + sg)];
          u += part[2 * (q * nseg + sg) + 1];
        }
        o.y[((a >> 1) + full) + q] = silu_mul_fast(g * o.scale, u * o.scale);
      }
    } else {
      for (int i = threadIdx.x; i < n - 2 * full; i += kCT) {
        const int q = i >> 1, w = i & 1;
        float v = 0.f;
        for (int sg = 0; sg < nseg; ++sg) v += part[2 * (q * nseg + sg) + w];
        epi_row<EPI>(o, a + 2 * full + i, v * o.scale);
      }
    }
  }
}

__device__ __forceinline__ void red_add_v4(float* p, float4 v) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// The down projection restricted to this block's columns [j0, j1) times its
// SwiGLU outputs hs[j - j0] (shared memory): a partial sum for each of the H
// rows, added into `out` (one of the copies of the current set) with
// vector atomic adds.  The columns arrive through the ring in the layout of
// DevModel::dcol_bytes; thread t owns rows 4t..4t+3 (H <= 4 consumer threads
// per row group).  Per Q8_0 block c: sum_j q[r][j] h_j over its columns, then
// times the f16 scale of (r, c) ("Eight kernels", q8_matvec, split by
// columns: the partial sums of the blocks add up to the row's dot product).
template <int FMT>
__device__ void down_cols(Cons& C, int j0, int j1, const float* hs, float* out) {
  const int H = C.m.H, t = threadIdx.x, lane = t & 31;
  const bool has = 4 * t < H;
  float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
  if (FMT == kFmtQ8) {
    const uint32_t sb = a16(2u * H);
    for (int c = j0 / 32; c * 32 < j1; ++c) {
      const int ja = max(j0, 32 * c), jb = min(j1, 32 * c + 32);
      mwait(C.r.full + C.r.n % kSlots, (C.r.n / kSlots) & 1u, C.err);
      const uint8_t* slot = slot_ptr(C.r);
      if (has) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const uint8_t* q = slot + sb + 4 * t;
        for (int j = ja; j < jb; ++j) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(q + static_cast<size_t>(j - ja) * H);
          const float hv = hs[j - j0];
          float f0, f1, f2, f3;
          i8x4_to_f32(w, f0, f1, f2, f3);
          acc.x = fmaf(f0, hv, acc.x);
          acc.y = fmaf(f1, hv, acc.y);
          acc.z = fmaf(f2, hv, acc.z);
          acc.w = fmaf(f3, hv, acc.w);
        }
        const uint2 sc = *reinterpret_cast<const uint2*>(slot + 8 * t);  // scales of rows 4t..4t+3
        tot.x = fmaf(acc.x, __half2float(__ushort_as_half(static_cast<unsigned short>(sc.x & 0xFFFFu))), tot.x);
        tot.y = fmaf(acc.y, __half2float(__ushort_as_half(static_cast<unsigned short>(sc.x >> 16))), tot.y);
        tot.z = fmaf(acc.z, __half2float(__ushort_as_half(static_cast<unsigned short>(sc.y & 0xFFFFu))), tot.z);
        tot.w = fmaf(acc.w, __half2float(__ushort_as_half(static_cast<unsigned short>(sc.y >> 16))), tot.w);
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(C.r.empty + C.r.n % kSlots)) : "memory");
      ++C.r.n;
    }
  } else {
    const int cpp = static_cast<int>(kSlotBytes / (2u * H));
    for (int a = j0; a < j1; a += cpp) {
      const int n = min(cpp, j1 - a);
      mwait(C.r.full + C.r.n % kSlots, (C.r.n / kSlots) & 1u, C.err);
      const uint8_t* slot = slot_ptr(C.r);
      if (has) {
        for (int k = 0; k < n; ++k) {
          const uint2 w = *reinterpret_cast<const uint2*>(slot + static_cast<size_t>(k) * 2u * H + 8 * t);
          const float hv = hs[a + k - j0];
          tot.x = fmaf(bf16_lo(w.x), hv, tot.x);
          tot.y = fmaf(bf16_hi(w.x), hv, tot.y);
          tot.z = fmaf(bf16_lo(w.y), hv, tot.z);
          tot.w = fmaf(bf16_hi(w.y), hv, tot.w);
        }
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(C.r.empty + C.r.n % kSlots)) : "memory");
      ++C.r.n;
    }
  }
  if (has && j0 < j1) red_add_v4(out + 4 * t, tot);
}

// Zero this block's share [e0, e1) of an array (plain stores).
__device__ __forceinline__ void zero_share(float* p, int e0, int e1) {
  for (int i = e0 + threadIdx.x; i < e1; i += kCT) p[i] = 0.f;
}

// Lane-strided words p[lane + 32 j], j < NJ, of tagged values other blocks
// write: poll until every one carries `tag`, then return the values.  The
// wait is bounded like the barrier waits; false (values undefined) if it gave
// up or another thread reported a fatal error.  Warp-uniform.
template <int NJ>
__device__ __forceinline__ bool poll_tagged(const uint64_t* p, uint32_t tag, float (&v)[NJ], uint32_t* err) {
  const int lane = threadIdx.x & 31;
  unsigned long long w[NJ];
  uint64_t t0 = 0;
  for (uint32_t spins = 0;; ++spins) {
#pragma unroll
    for (int j = 0; j < NJ; ++j) w[j] = ld_tagged(p + lane + 32 * j);
    bool ok = true;
#pragma unroll
    for (int j = 0; j < NJ; ++j) ok = ok && static_cast<uint32_t>(w[j] >> 32) == tag;
    if (__all_sync(0xFFFFFFFFu, ok)) break;
    if (spins == 0) t0 = global_timer_ns();
    if ((spins & 15u) == 15u) {
      int bad = 0;
      if (lane == 0) {
        if (ld_volatile_u32(err) & kFatal) bad = 1;
        else if (global_timer_ns() - t0 > kWaitLimitNs) {
          atomicOr(err, kErrGridBarrier);
          bad = 1;
        }
      }
      if (__shfl_sync(0xFFFFFFFFu, bad, 0)) return false;
    }
  }
#pragma unroll
  for (int j = 0; j < NJ; ++j) v[j] = __uint_as_float(static_cast<uint32_t>(w[j]));
  return true;
}

// Constants of the attention phase a lane needs (QK-norm gains and the RoPE
// (cos, sin) pairs of the current position), loaded before the barrier wait.
struct AttnPre {
  float qg[4], kg[4];
  float2 cs[2];
  uint32_t tag;  // the tag this layer's projections are written with
};

__device__ __forceinline__ void load_attn_pre(AttnPre& p, const DevModel& m, const DevLayer& L,
                                              int pos) {
  const int lane = threadIdx.x & 31;
  const int nj = m.hd / 32;
  const float2* rope = m.rope + static_cast<size_t>(pos) * (m.hd / 2);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    p.qg[j] = (m.qk_norm && j < nj) ? __ldg(L.q_norm + lane + 32 * j) : 1.f;
    p.kg[j] = (m.qk_norm && j < nj) ? __ldg(L.k_norm + lane + 32 * j) : 1.f;
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) p.cs[j] = j < nj / 2 ? __ldg(rope + lane + 32 * j) : make_float2(1.f, 0.f);
}

// Per-head RMSNorm (optional) and half-split RoPE of one head held as
// lane-strided elements e_j = lane + 32 j ("Eight kernels", rms_norm_row and
// rope_row), with the gains and rotation pairs already in registers.
template <int HD>
__device__ __forceinline__ void norm_rope_regs(float (&v)[HD / 32], const float* g, bool norm,
                                               const float2* cs, float eps) {
  constexpr int NJ = HD / 32;
  if (norm) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) ss = fmaf(v[j], v[j], ss);
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / static_cast<float>(HD) + eps);
#pragma unroll
    for (int j = 0; j < NJ; ++j) v[j] = v[j] * inv * g[j];
  }
#pragma unroll
  for (int j = 0; j < NJ / 2; ++j) {
    const float u = v[j], w = v[j + NJ / 2];
    v[j] = u * cs[j].x - w * cs[j].y;
    v[j + NJ / 2] = u * cs[j].y + w * cs[j].x;
  }
}

// Attention for item (g, c): queries of kv group g against the chunk's cached
// rows (streamed through the ring) plus the new row; online softmax; the last
// chunk of the group to finish combines all chunks ("Eight kernels",
// attention_decode, as a split-K flash decode).
template <int HD, int G>
__device__ void attn_item(Cons& C, int layer, int g, int c, int pos, int t0, int t1, const AttnPre& pre) {
  constexpr int NJ = HD / 32, DPL = HD / 32;
  const DevModel& m = C.m;
  const DevSeq& s = C.s;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* qs = C.scr;               // [G][HD]
  float* knew = qs + G * HD;       // [HD]
  float* vnew = knew + HD;         // [HD]
  float* wst = vnew + HD;          // [kCW][G][HD + 2], then the group's partials
  const bool has_new = t0 <= pos && pos < t1;
  const int tc = min(t1, pos);     // cached rows end
  if (warp < G) {
    const int h = g * G + warp;
    float v[NJ];
    poll_tagged<NJ>(s.qkv_tag + h * HD, pre.tag, v, C.err);  // a failed wait leaves the error bit for later waits
    norm_rope_regs<HD>(v, pre.qg, m.qk_norm != 0, pre.cs, m.eps);
#pragma unroll
    for (int j = 0; j < NJ; ++j) qs[warp * HD + lane + 32 * j] = v[j];
  } else if (warp == kCW - 1 && has_new) {
    // the new row: QK-norm + RoPE on k, append k and v to the cache
    // ("Eight kernels", append_kv)
    float kv[NJ], vv[NJ];
    if (poll_tagged<NJ>(s.qkv_tag + m.qw + g * HD, pre.tag, kv, C.err))
      poll_tagged<NJ>(s.qkv_tag + m.qw + m.kvw + g * HD, pre.tag, vv, C.err);
    norm_rope_regs<HD>(kv, pre.kg, m.qk_norm != 0, pre.cs, m.eps);
    const size_t row = ((static_cast<size_t>(layer) * m.nkv + g) * m.max_seq + pos) * HD;
    if (m.kv16) {  // rounded to binary16 as it enters the cache, and used rounded
      __half* kh = reinterpret_cast<__half*>(s.kcache) + row;
      __half* vh = reinterpret_cast<__half*>(s.vcache) + row;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const __half k16 = __float2half_rn(kv[j]), v16 = __float2half_rn(vv[j]);
        kh[lane + 32 * j] = k16;
        vh[lane + 32 * j] = v16;
        kv[j] = __half2float(k16);
        vv[j] = __half2float(v16);
      }
    } else {
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        s.kcache[row + lane + 32 * j] = kv[j];
        s.vcache[row + lane + 32 * j] = vv[j];
      }
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      knew[lane + 32 * j] = kv[j];
      vnew[lane + 32 * j] = vv[j];
    }
    fence_proxy_async_global();  // later bulk copies read this row
  }
  csync();
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
  // a row's K and V elements of this lane, from f32 or f16 rows
  auto load_row = [&](const void* kr, const void* vr, bool half, float (&kf)[DPL], float (&vf)[DPL]) {
    if (half) {
      const __half* kh = static_cast<const __half*>(kr) + lane * DPL;
      const __half* vh = static_cast<const __half*>(vr) + lane * DPL;
#pragma unroll
      for (int e = 0; e < DPL; e += 2) {
        const float2 k2 = __half22float2(*reinterpret_cast<const __half2*>(kh + e));
        const float2 v2 = __half22float2(*reinterpret_cast<const __half2*>(vh + e));
        kf[e] = k2.x; kf[e + 1] = k2.y;
        vf[e] = v2.x; vf[e + 1] = v2.y;
      }
    } else if constexpr (DPL == 4) {
      const float4 k4 = *reinterpret_cast<const float4*>(static_cast<const float*>(kr) + lane * 4);
      const float4 v4 = *reinterpret_cast<const float4*>(static_cast<const float*>(vr) + lane * 4);
      kf[0] = k4.x; kf[1] = k4.y; kf[2] = k4.z; kf[3] = k4.w;
      vf[0] = v4.x; vf[1] = v4.y; vf[2] = v4.z; vf[3] = v4.w;
    } else {
      const float2 k2 = *reinterpret_cast<const float2*>(static_cast<const float*>(kr) + lane * 2);
      const float2 v2 = *reinterpret_cast<const float2*>(static_cast<const float*>(vr) + lane * 2);
      kf[0] = k2.x; kf[1] = k2.y;
      vf[0] = v2.x; vf[1] = v2.y;
    }
  };
  auto row_update = [&](const float (&kf)[DPL], const float (&vf)[DPL]) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) d = fmaf(qv[hh][e], kf[e], d);
      const float sc = warp_sum(d) * m.attn_scale;
      if (sc > mm[hh]) {
        const float corr = __expf(mm[hh] - sc);
        mm[hh] = sc;
        ll[hh] = ll[hh] * corr + 1.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) oo[hh][e] = fmaf(oo[hh][e], corr, vf[e]);
      } else {
        const float p = __expf(sc - mm[hh]);
        ll[hh] += p;
#pragma unroll
        for (int e = 0; e < DPL; ++e) oo[hh][e] = fmaf(p, vf[e], oo[hh][e]);
      }
    }
  };
  const bool kv16 = m.kv16 != 0;
  const int esz = kv16 ? 2 : 4;
  const int rpp = kv_rows_per_piece(HD, esz);
  for (int a = t0; a < tc; a += rpp) {
    const int n = min(rpp, tc - a);
    mwait(C.r.full + C.r.n % kSlots, (C.r.n / kSlots) & 1u, C.err);
    const uint8_t* Ks = slot_ptr(C.r);
    const uint8_t* Vs = Ks + static_cast<size_t>(rpp) * HD * esz;
    int t = warp;
    for (; t + kCW < n; t += 2 * kCW) {  // two rows at a time: both scores before one softmax update
      float kf[DPL], vf[DPL], kg[DPL], vg[DPL];
      load_row(Ks + static_cast<size_t>(t) * HD * esz, Vs + static_cast<size_t>(t) * HD * esz, kv16, kf, vf);
      load_row(Ks + static_cast<size_t>(t + kCW) * HD * esz, Vs + static_cast<size_t>(t + kCW) * HD * esz, kv16, kg, vg);
      float d1[G], d2[G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        d1[hh] = 0.f;
        d2[hh] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
          d1[hh] = fmaf(qv[hh][e], kf[e], d1[hh]);
          d2[hh] = fmaf(qv[hh][e], kg[e], d2[hh]);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          d1[hh] += __shfl_xor_sync(0xFFFFFFFFu, d1[hh], o);
          d2[hh] += __shfl_xor_sync(0xFFFFFFFFu, d2[hh], o);
        }
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float s1 = d1[hh] * m.attn_scale, s2 = d2[hh] * m.attn_scale;
        const float mn = fmaxf(mm[hh], fmaxf(s1, s2));
        const float corr = __expf(mm[hh] - mn), p1 = __expf(s1 - mn), p2 = __expf(s2 - mn);
        mm[hh] = mn;
        ll[hh] = fmaf(ll[hh], corr, p1 + p2);
#pragma unroll
        for (int e = 0; e < DPL; ++e) oo[hh][e] = fmaf(oo[hh][e], corr, fmaf(p1, vf[e], p2 * vg[e]));
      }
    }
    if (t < n) {
      float kf[DPL], vf[DPL];
      load_row(Ks + static_cast<size_t>(t) * HD * esz, Vs + static_cast<size_t>(t) * HD * esz, kv16, kf, vf);
      row_update(kf, vf);
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(C.r.empty + C.r.n % kSlots)) : "memory");
    ++C.r.n;
  }
  if (has_new && warp == ((tc - t0) % kCW)) {
    float kf[DPL], vf[DPL];
    load_row(knew, vnew, false, kf, vf);
    row_update(kf, vf);
  }
  // merge the warps' states
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
  csync();
  // per head, once (one warp each): the chunk's max M over the warps, their
  // weights f_w = exp(m_w - M) and the chunk's sum; written over qs, which
  // every warp finished reading before its rows
  float* fw = qs;  // [G][kCW] weights, then [G][2] (M, sum)
  if (warp < G) {
    const float mw = lane < kCW ? wst[(lane * G + warp) * stride + HD] : -INFINITY;
    const float M = warp_max(mw);
    const float f = (lane < kCW && mw != -INFINITY) ? __expf(mw - M) : 0.f;
    const float Ls = warp_sum(lane < kCW ? f * wst[(lane * G + warp) * stride + HD + 1] : 0.f);
    if (lane < kCW) fw[warp * kCW + lane] = f;
    if (lane == 0) {
      fw[G * kCW + 2 * warp] = M;
      fw[G * kCW + 2 * warp + 1] = Ls;
    }
  }
  csync();
  for (int idx = threadIdx.x; idx < G * HD; idx += kCT) {
    const int hh = idx / HD, d = idx - hh * HD;
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) O = fmaf(fw[hh * kCW + w], wst[(w * G + hh) * stride + d], O);
    const int h = g * G + hh;
    s.part_o[(static_cast<size_t>(h) * m.n_chunks + c) * HD + d] = O;
    if (d == 0) {
      s.part_ml[(static_cast<size_t>(h) * m.n_chunks + c) * 2] = fw[G * kCW + 2 * hh];
      s.part_ml[(static_cast<size_t>(h) * m.n_chunks + c) * 2 + 1] = fw[G * kCW + 2 * hh + 1];
    }
  }
}

// Combine group g's chunk partials by log-sum-exp ("Eight kernels",
// attention_decode, as a split-K flash decode) into the matvec input (the
// padded layout) of the group's O column slice: xin holds o of the group's
// heads, G * head_dim values.
template <int HD>
__device__ void group_combine(Cons& C, int g, int G) {
  const DevModel& m = C.m;
  const DevSeq& s = C.s;
  const int NC = m.n_chunks;
  float* po = C.scr;                      // [G][NC][HD]
  float* pml = po + G * NC * HD;          // [G][NC][2]
  // every partial is requested before any is stored (one L2 round trip):
  // the partials are at most 24 KB (the engine caps the chunk count), so at
  // most kCombineLoads float4 per thread
  const int n4 = G * NC * HD / 4, nml = G * NC * 2;
  const float4* src_o = reinterpret_cast<const float4*>(s.part_o + static_cast<size_t>(g) * G * NC * HD);
  const float* src_ml = s.part_ml + static_cast<size_t>(g) * G * NC * 2;
  constexpr int kCombineLoads = 4;
  float4 r[kCombineLoads];
#pragma unroll
  for (int k = 0; k < kCombineLoads; ++k) {
    const int i = threadIdx.x + k * kCT;
    r[k] = i < n4 ? __ldcg(src_o + i) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ml[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = threadIdx.x + k * kCT;
    ml[k] = i < nml ? __ldcg(src_ml + i) : 0.f;
  }
#pragma unroll
  for (int k = 0; k < kCombineLoads; ++k) {
    const int i = threadIdx.x + k * kCT;
    if (i < n4) reinterpret_cast<float4*>(po)[i] = r[k];
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = threadIdx.x + k * kCT;
    if (i < nml) pml[i] = ml[k];
  }
  csync();
  // chunk weights exp(m_c - M) / L of every head, once: one warp per head
  float* wts = pml + G * NC * 2;          // [G][NC]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < G) {
    float M = -INFINITY;
    for (int cc = lane; cc < NC; cc += 32) M = fmaxf(M, pml[(warp * NC + cc) * 2]);
    M = warp_max(M);
    float den = 0.f;
    for (int cc = lane; cc < NC; cc += 32) {
      const float mc = pml[(warp * NC + cc) * 2];
      const float f = mc == -INFINITY ? 0.f : __expf(mc - M);
      wts[warp * NC + cc] = f;
      den = fmaf(f, pml[(warp * NC + cc) * 2 + 1], den);
    }
    den = warp_sum(den);
    __syncwarp();
    for (int cc = lane; cc < NC; cc += 32) wts[warp * NC + cc] /= den;
  }
  csync();
  for (int idx = threadIdx.x; idx < G * HD; idx += kCT) {
    const int hh = idx / HD, d = idx - hh * HD;
    float num = 0.f;
    for (int cc = 0; cc < NC; ++cc) num = fmaf(wts[hh * NC + cc], po[(hh * NC + cc) * HD + d], num);
    C.xin[xpad(C.fmt, idx)] = num;
  }
  csync();
}


// One kernel per (weight format, head_dim, q heads per kv head), so that each
// holds only its own attention variant.
template <int FMT, int HD, int GQ>
__device__ void run_consumers(Cons& C, int n_steps, int full_from, uint32_t pos0) {
  const DevModel& m = C.m;
  const DevSeq& s = C.s;
  const int b = blockIdx.x, nb = gridDim.x;
  DevBarrier* bar = s.bar;
  unsigned long long epoch = s.bar->epoch;  // barriers completed before this launch
  const int G = m.nq / m.nkv;
  auto arrive = [&]() {
    gb_arrive(bar);
    ++epoch;
  };
  auto wait = [&]() { return gb_wait(bar, epoch * static_cast<unsigned long long>(nb), C.err); };
  // the plan in shared memory: indexed by a loop variable, a local copy would
  // live in local memory, which misses the small L1 left beside the
  // shared-memory carve-out on every layer
  __shared__ Plan s_pl;
  if (threadIdx.x == 0) s_pl = make_plan(m, b, nb);
  csync();
  const Plan& pl = s_pl;
  const int v0 = pl.v0, v1 = pl.v1;
  // each counter on its own 128-byte line: groups do not contend
  DevBarrier* ga = pl.grp >= 0 ? s.gbar + 16 * pl.grp : nullptr;  // its epoch: the group's layers so far (kept across launches)
  DevBarrier* gb = pl.grp >= 0 ? ga + 8 : nullptr;                 // the group's attention partials are written
  unsigned long long gepoch = pl.grp >= 0 ? ga->epoch : 0ull;      // the group's layers before this launch
  // FFN phases of this launch: phase k adds its down-projection partial sums
  // into set k & 1 of xacc (kAccCopies copies, block b adding into copy
  // b % kAccCopies, to spread the atomic adds) and clears this block's share of the other set, which the
  // next FFN phase sums into after at least two more grid barriers; readers
  // of set k (the next layer's input, or the lm_head's) finish before the
  // grid barrier that starts FFN phase k + 1.  Set 0 is cleared here.
  const int H = m.H;
  const int rpp_h = rows_per_piece(m.row_bytes_h), rpp_gh = rows_per_piece(m.row_bytes_gh);  // rows per ring piece
  const int rpp_gu = rows_per_piece_all(m.row_bytes_h);
  int kph = 0;
  zero_share(s.xacc, pl.zx0, pl.zx1);
  zero_share(s.opart, pl.zo0, pl.zo1);
  // the O products of the first layer are added into opart set 0 by blocks of
  // every group before any later grid barrier: the clearing must be visible
  // first (one extra grid barrier per launch)
  arrive();
  if (!wait()) return;
  for (int step = 0; step < n_steps; ++step) {
    const uint32_t pos = pos0 + step;
    if (pos >= static_cast<uint32_t>(m.max_seq)) {
      if (b == 0 && threadIdx.x == 0) atomicOr(C.err, kErrCapacity);
      break;
    }
    if (step > 0 && !wait()) return;  // the previous step's token is written
    int tok = (step == 0 && s.tok_in >= 0) ? s.tok_in : __ldcg(s.tokens + pos);
    if (step == 0 && s.tok_in >= 0 && b == 0 && threadIdx.x == 0) s.tokens[pos] = s.tok_in;  // the history
    int ct0 = 0, ct1 = 0;  // this block's attention chunk of the step's pos + 1 rows
    if (pl.chunk >= 0) chunk_range(static_cast<int>(pos) + 1, m.n_chunks, pl.chunk, ct0, ct1);
    if (tok < 0 || tok >= m.V) {
      if (threadIdx.x == 0) atomicOr(C.err, kErrBadToken);
      tok = 0;
    }
    for (int l = 0; l < m.n_layers; ++l) {
      const DevLayer L = m.layers[l];  // pointers read before any wait
      MvOut o{};
      Gain gain;
      load_gain(gain, L.attn_norm, m.H);
      // ---- RMSNorm + the group's Q, K, V rows ----
      if (l == 0) {
        csync();
        if (FMT == kFmtQ8) {
          const uint8_t* row = m.embed + static_cast<size_t>(tok) * m.row_bytes_h;
          const __half* sc = reinterpret_cast<const __half*>(row + m.H);
          for (int i = threadIdx.x; i < m.H; i += kCT)
            C.xraw[i] = __half2float(sc[i >> 5]) * static_cast<float>(static_cast<int8_t>(row[i]));
        } else {
          const uint16_t* row = reinterpret_cast<const uint16_t*>(m.embed + static_cast<size_t>(tok) * m.row_bytes_h);
          for (int i = threadIdx.x; i < m.H; i += kCT) C.xraw[i] = __uint_as_float(static_cast<uint32_t>(row[i]) << 16);
        }
        csync();
        o.scale = to_xin_norm(C, C.xraw, m.H, gain);
      } else {
        if (!wait()) return;
        o.scale = load_norm_sum(C, s.xacc + ((kph - 1) & 1) * kAccCopies * H, kAccCopies, H, gain);
      }
      // the group's Q, K and V rows as tagged words: the attention blocks of
      // the group poll exactly the rows they need, with no barrier between
      o.ytag = s.qkv_tag;
      o.tag = static_cast<uint32_t>(gepoch + 1);
      for (int i = 0; i < 3; ++i)
        if (pl.qr0[i] < pl.qr1[i]) mv_phase<FMT, kEpiTagged, false>(C, m.row_bytes_h, rpp_h, m.H, pl.qr0[i], pl.qr1[i], o);
      load_gain(gain, L.ffn_norm, m.H);  // for the gate/up phase
      if (pl.grp >= 0) {
        const unsigned long long tgt = (gepoch + 1) * static_cast<unsigned long long>(pl.bpg);
        // ---- QK-norm + RoPE + append + attention chunk ----
        if (pl.chunk >= 0) {
          AttnPre pre;
          load_attn_pre(pre, m, L, static_cast<int>(pos));
          pre.tag = static_cast<uint32_t>(gepoch + 1);
          attn_item<HD, GQ>(C, l, pl.grp, pl.chunk, pos, ct0, ct1, pre);
        }
        gb_arrive(gb);
        ++gepoch;
        // ---- combine the group's chunks + its O column slice ----
        if (!gb_wait(gb, tgt, C.err)) return;
        group_combine<HD>(C, pl.grp, G);
        o.scale = 1.f;
        // kEpiAtomicAdd: the groups' products of a row meet in one sum
        o.y = s.opart + static_cast<size_t>(kph & 1) * m.H;
        mv_phase<FMT, kEpiAtomicAdd, (GQ * HD) / epc_of(FMT) <= 16>(C, m.row_bytes_gh, rpp_gh, G * m.hd, pl.o0, pl.o1, o);
      }
      arrive();
      // ---- residual + RMSNorm + gate/up + SwiGLU, then the down projection
      //      over this block's SwiGLU outputs, summed into xacc ----
      if (!wait()) return;
      o.scale = load_norm_sum(C, s.opart + static_cast<size_t>(kph & 1) * m.H, 1, H, gain);
      zero_share(s.opart + static_cast<size_t>((kph + 1) & 1) * m.H, pl.zo0, pl.zo1);
      const int j0 = pl.g0 / 2, j1 = pl.g1 / 2;
      o.y = C.scr - j0;  // h[j] of this block's rows, in shared memory at scr[j - j0]
      mv_phase<FMT, kEpiSwiGLU, false, true>(C, m.row_bytes_h, rpp_gu, H, pl.g0, pl.g1, o);
      csync();
      down_cols<FMT>(C, j0, j1, C.scr, s.xacc + (kph & 1) * kAccCopies * H + (b % kAccCopies) * H);
      zero_share(s.xacc + ((kph + 1) & 1) * kAccCopies * H, pl.zx0, pl.zx1);
      ++kph;
      arrive();
    }
    if (step >= full_from) {
      // ---- final RMSNorm + lm_head + argmax ----
      Gain gain;
      load_gain(gain, m.out_norm, m.H);
      if (!wait()) return;
      MvOut o{};
      o.scale = load_norm_sum(C, s.xacc + ((kph - 1) & 1) * kAccCopies * H, kAccCopies, H, gain);
      o.y = s.logits;
      o.bv = -INFINITY;
      o.bi = INT_MAX;
      mv_phase<FMT, kEpiArgmax, false>(C, m.row_bytes_h, rpp_h, m.H, v0, v1, o);
      // block candidate -> global candidates -> the last block picks the winner
      warp_argmax(o.bv, o.bi);
      float* redv = C.red + 32;                         // clear of the norm partials
      int* redi = reinterpret_cast<int*>(C.red + 48);
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
      if (lane == 0) {
        redv[warp] = o.bv;
        redi[warp] = o.bi;
      }
      csync();
      __shared__ uint32_t s_last;
      if (threadIdx.x == 0) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int w = 0; w < kCW; ++w) argmax_merge(bv, bi, redv[w], redi[w]);
        s.amax_v[b] = bv;
        s.amax_i[b] = bi;
        __threadfence();
        const uint32_t old = atomicAdd(s.amax_count, 1u);
        s_last = old == static_cast<uint32_t>(nb) - 1u;
        if (s_last) __threadfence();
      }
      csync();
      if (s_last) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int k = threadIdx.x; k < nb; k += kCT) argmax_merge(bv, bi, __ldcg(s.amax_v + k), __ldcg(s.amax_i + k));
        warp_argmax(bv, bi);
        csync();  // every warp has read redv / redi above
        if (lane == 0) {
          redv[warp] = bv;
          redi[warp] = bi;
        }
        csync();
        if (threadIdx.x == 0) {
          float v = -INFINITY;
          int i = INT_MAX;
          for (int w = 0; w < kCW; ++w) argmax_merge(v, i, redv[w], redi[w]);
          int next = i;
          if (i == INT_MAX) {
            atomicOr(C.err, kErrAllNaN);
            next = -1;
          }
          if (pos + 1 <= static_cast<uint32_t>(m.max_seq)) s.tokens[pos + 1] = next;
          s.state->last = next;
          s.state->pos = pos + 1;
          s.state->steps += 1;
          *s.amax_count = 0u;
        }
      }
      arrive();
    } else if (b == 0 && threadIdx.x == 0) {
      s.state->pos = pos + 1;
      s.state->steps += 1;
    }
  }
  if (b == 0 && threadIdx.x == 0) s.bar->epoch = epoch;
  if (pl.grp >= 0 && pl.j == 0 && threadIdx.x == 0) ga->epoch = gepoch;
}

template <int FMT, int HD, int GQ>
__global__ void __launch_bounds__(kThreads, 1)
    k_persist(DevModel m, DevSeq s, int n_steps, int full_from) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const PLayout L = playout(m);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
  uint64_t* empty = full + kSlots;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kCW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t pos0 = __ldcg(&s.state->pos);
  Ring ring{sm + L.ring, full, empty, 0};
  if (threadIdx.x >= kCT) {
    if (threadIdx.x == kCT) run_producer(m, s, n_steps, full_from, pos0, ring);
    return;
  }
  Cons C(m, s);
  C.r = ring;
  C.xraw = reinterpret_cast<float*>(sm + L.xraw);
  C.xin = reinterpret_cast<float*>(sm + L.xin);
  C.scr = reinterpret_cast<float*>(sm + L.scratch);
  C.red = reinterpret_cast<float*>(sm + L.red);
  C.rsel = 0;
  C.psel = 0;
  C.err = &s.state->err;
  C.fmt = FMT;
  C.inv_h = 1.0f / static_cast<float>(m.H);
  run_consumers<FMT, HD, GQ>(C, n_steps, full_from, pos0);
}

template <int FMT, int HD>
const void* persist_fn_g(int G) {
  switch (G) {
    case 1: return reinterpret_cast<const void*>(&k_persist<FMT, HD, 1>);
    case 2: return reinterpret_cast<const void*>(&k_persist<FMT, HD, 2>);
    case 3: return reinterpret_cast<const void*>(&k_persist<FMT, HD, 3>);
    default: return reinterpret_cast<const void*>(&k_persist<FMT, HD, 4>);
  }
}

}  // namespace
}  // namespace tqd
