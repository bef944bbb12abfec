// Seeded sampling of the next token from a step's logits ("Metal LLM decode",
// the sampled arm of the batched prefill+decode section: temperature, top_k,
// top_p, min_p, repeat / presence / frequency penalties and a seed;
// temperature <= 0 falls back to the greedy token and top_k = 1 reproduces
// it).  With 1 <= top_k <= kSamplePartK the draw takes two passes
// (k_sample_part keeps each vocabulary slice's first top_k under the
// penalties, k_sample merges them and runs the list path below); otherwise,
// and where the merge cannot decide, one block per sequence does everything,
// in this order:
//   1. penalties on the distinct tokens among the sequence's inputs (counted
//      in a per-sequence array the block leaves zeroed), each an f32
//      operation: a = l > 0 ? l / r : l * r; a -= presence; a -= frequency * c;
//      NaN -> -inf; the penalised logits go to a per-sequence array;
//   2. the order: penalised logit l descending, index ascending.  Division by
//      T > 0 keeps that order, and ranking before the division keeps top_k = 1
//      equal to the greedy token where l / T merges two adjacent logits;
//   3. top_k: the first k tokens of that order;
//   4. top_p: of those, in that order, the shortest prefix whose mass reaches
//      p of their mass;
//   5. min_p: z - z_max >= ln(min_p), z = l / T in f32 (f32 difference; the
//      log taken on the host);
//   6. draw: u = the top 24 bits of splitmix64's output at the drawn token's
//      position, times 2^-24; the token is the first kept one in index order
//      whose running mass exceeds u times the kept mass.
// Masses are exp(z - z_max) in f32, carried as integers in units of 2^-32 of
// the most likely token's, so every sum is exact and independent of order and
// the draw is deterministic.  When l_max / T overflows f32 (the limit T -> 0)
// the draw is the greedy token of the penalised logits.  A boundary (steps 3,
// 4) is found by a histogram of the values over [l_min, l_max], then an exact
// sort of the boundary bin's tokens (a zoom into the bin when it holds too
// many), ties in index order.
#include <climits>

#include "tqd_internal.h"

namespace tqd {
namespace {

constexpr int kSThreads = 512;
constexpr int kSWarps = kSThreads / 32;
constexpr int kSBins = 1024;                // value bins of a boundary search
constexpr int kSCand = 4096;                // tokens sorted exactly in shared memory
constexpr float kFix = 4294967296.0f;       // 2^32: the mass of the most likely token
constexpr unsigned long long kGolden = 0x9E3779B97F4A7C15ull;

struct SampleSm {
  unsigned long long hw[kSBins];    // weight per bin
  unsigned int hc[kSBins];          // tokens per bin
  unsigned long long cand[kSCand];  // (order key << 32) | (2^32 - 1 - index)
  unsigned long long wred[kSWarps];
  float fa[kSWarps], fb[kSWarps];
  unsigned int ncand;
  int bin;
  unsigned long long above_bin, need, r64;
  unsigned int cnt_bin;
  float zb;
  int ib;
};

// Unsigned key ordered like the float.
__device__ __forceinline__ uint32_t order_key(float z) {
  const uint32_t u = __float_as_uint(z);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// splitmix64's output function (Steele, Lea and Flood, 2014).
__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ unsigned long long wfix(float z, float zmax) {
  return __float2ull_rz(__fmul_rn(expf(__fsub_rn(z, zmax)), kFix));
}

// The mass of a token with penalised logit l: z = l / T, weight exp(z - z_max).
struct LWeight {
  float temp, zmax;
  __device__ unsigned long long operator()(float l) const { return wfix(__fdiv_rn(l, temp), zmax); }
};

// A token v of penalised logit l is kept when it passes every stage set so far.
struct Keep {
  float kz;
  int ki;      // top_k: l > kz, or l == kz and v <= ki
  float pz;
  int pi;      // top_p: the same
  float temp;
  float zmax;
  float lnmp;  // min_p: l / T - zmax >= lnmp (-inf when off)
  __device__ bool operator()(int v, float l) const {
    return (l > kz || (l == kz && v <= ki)) && (l > pz || (l == pz && v <= pi)) &&
           __fsub_rn(__fdiv_rn(l, temp), zmax) >= lnmp;
  }
};

__device__ unsigned long long block_sum(unsigned long long x, SampleSm& sm) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.wred[threadIdx.x >> 5] = x;
  __syncthreads();
  unsigned long long t = 0;
  for (int i = 0; i < kSWarps; ++i) t += sm.wred[i];
  return t;
}

// (max of a, min of b) over the block
__device__ void block_maxmin(float& a, float& b, SampleSm& sm) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    b = fminf(b, __shfl_xor_sync(0xFFFFFFFFu, b, o));
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    sm.fa[threadIdx.x >> 5] = a;
    sm.fb[threadIdx.x >> 5] = b;
  }
  __syncthreads();
  a = sm.fa[0];
  b = sm.fb[0];
  for (int i = 1; i < kSWarps; ++i) {
    a = fmaxf(a, sm.fa[i]);
    b = fminf(b, sm.fb[i]);
  }
}

// f(v, z[v]) for every v < V.  z is padded to whole float4 groups; a thread
// takes groups t, t + T, t + 2T, t + 3T per round, four loads in flight.
template <class F>
__device__ __forceinline__ void each4(const float* z, int V, F&& f) {
  const int n4 = (V + 3) >> 2;
  const float4* z4 = reinterpret_cast<const float4*>(z);
  for (int g0 = threadIdx.x; g0 < n4; g0 += 4 * kSThreads) {
    float4 q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * kSThreads;
      q[u] = g < n4 ? z4[g] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * kSThreads;
      if (g < n4) {
        const int v = 4 * g;
        f(v, q[u].x);
        if (v + 1 < V) f(v + 1, q[u].y);
        if (v + 2 < V) f(v + 2, q[u].z);
        if (v + 3 < V) f(v + 3, q[u].w);
      }
    }
  }
}

// The smallest v < V whose running weight (over 0..v, index order) exceeds
// thresh, with that running weight in sm.r64; V when the total does not.
// A thread takes four consecutive float4 groups of each chunk.
template <class Wt>
__device__ int first_over(const float* z, int V, Wt weight, unsigned long long thresh, SampleSm& sm) {
  constexpr int G = 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n4 = (V + 3) >> 2;
  const float4* z4 = reinterpret_cast<const float4*>(z);
  unsigned long long run = 0;
  for (int c0 = 0; c0 < n4; c0 += kSThreads * G) {
    const int g0 = c0 + static_cast<int>(threadIdx.x) * G;
    float q[4 * G];
#pragma unroll
    for (int u = 0; u < G; ++u) {
      const float4 f4 = g0 + u < n4 ? z4[g0 + u] : make_float4(0.f, 0.f, 0.f, 0.f);
      q[4 * u] = f4.x;
      q[4 * u + 1] = f4.y;
      q[4 * u + 2] = f4.z;
      q[4 * u + 3] = f4.w;
    }
    unsigned long long s = 0;
#pragma unroll
    for (int e = 0; e < 4 * G; ++e) {
      const int v = 4 * g0 + e;
      if (v < V) s += weight(v, q[e]);
    }
    unsigned long long x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) sm.wred[warp] = x;
    __syncthreads();
    unsigned long long wpre = 0, tot = 0;
    for (int i = 0; i < kSWarps; ++i) {
      const unsigned long long t = sm.wred[i];
      if (i < warp) wpre += t;
      tot += t;
    }
    if (run + tot > thresh) {  // the crossing is in this chunk, in one thread's elements
      const unsigned long long ex = run + wpre + x - s;
      if (ex <= thresh && thresh < ex + s) {
        unsigned long long acc = ex;
        for (int e = 0; e < 4 * G; ++e) {
          const int v = 4 * g0 + e;
          if (v >= V) break;
          acc += weight(v, q[e]);
          if (acc > thresh) {
            sm.ib = v;
            sm.r64 = acc;
            break;
          }
        }
      }
      __syncthreads();
      return sm.ib;
    }
    run += tot;
  }
  return V;
}

// The float an order key came from.
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Bitonic sort of sm.cand[0, P) (P a power of two), descending or ascending.
__device__ void sort_cand(int P, bool descending, SampleSm& sm) {
  for (int k = 2; k <= P; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += kSThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = sm.cand[i], b = sm.cand[ixj];
          if ((((i & k) == 0) == descending) ? (a < b) : (a > b)) {
            sm.cand[i] = b;
            sm.cand[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
}

// The first i < n at which the running weight (over 0..i) reaches thr, and
// the running weight there (sm.r64); n - 1 if it never does.  Warp 0 scans
// contiguous slices of the list; the result is broadcast.
template <class Wt>
__device__ int list_first_ge(int n, Wt weight_at, unsigned long long thr, SampleSm& sm) {
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) == 0) {
    const int per = (n + 31) / 32, i0 = min(n, lane * per), i1 = min(n, i0 + per);
    unsigned long long s = 0;
    for (int i = i0; i < i1; ++i) s += weight_at(i);
    unsigned long long x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, x >= thr);
    const int L = ball ? __ffs(ball) - 1 : 31;
    if (lane == L) {
      unsigned long long acc = x - s;
      int found = n - 1;
      for (int i = i0; i < i1; ++i) {
        acc += weight_at(i);
        if (acc >= thr) {
          found = i;
          break;
        }
      }
      if (!ball) acc = x;
      sm.ib = found;
      sm.r64 = acc;
    }
  }
  __syncthreads();
  const int r = sm.ib;
  __syncthreads();
  return r;
}

struct Sel {
  float zb;
  int ib;                   // the boundary: z > zb, or z == zb and index <= ib
  unsigned long long wsel;  // the selected tokens' weight (mass mode)
};

// The first `need` weight units of the tokens that pass `in`, in the order
// (z descending, index ascending), as a boundary.  need = need_abs if
// nonzero, else ceil(frac * the set's weight) (at least 1).  hi: the set's
// largest value; lo: a lower bound of its finite values.  A histogram of the
// values in [lo, hi] finds the bin where the running weight reaches need; the
// bin's tokens are sorted exactly, or, when too many, the search zooms into
// the bin's own range; a single remaining value is cut in index order.
template <class In, class Wt>
__device__ Sel select_top(const float* z, int V, In in, Wt weight, unsigned long long need_abs, float frac,
                          float hi, float lo, SampleSm& sm) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  unsigned long long above = 0;  // weight of the set's tokens above hi
  unsigned long long need = need_abs;
  if (!(hi > lo) && need == 0ull) {  // one value only: the set's weight directly
    unsigned long long w = 0;
    each4(z, V, [&](int v, float zv) {
      if (zv > -INFINITY && in(v, zv)) w += weight(v, zv);
    });
    w = block_sum(w, sm);
    need = static_cast<unsigned long long>(ceil(static_cast<double>(frac) * static_cast<double>(w)));
    need = need < 1ull ? 1ull : (need > w ? w : need);
  }
  for (int round = 0; round < 8 && hi > lo; ++round) {
    const float inv_w = __fdiv_rn(static_cast<float>(kSBins), __fsub_rn(hi, lo));
    if (!(inv_w > 0.f) || !(inv_w < INFINITY)) break;
    auto bin_of = [&](float zv) {  // monotone in zv: the same value always lands in the same bin
      const float q = __fmul_rn(__fsub_rn(hi, zv), inv_w);
      return q >= static_cast<float>(kSBins - 1) ? kSBins - 1 : (q > 0.f ? static_cast<int>(q) : 0);
    };
    for (int i = t; i < kSBins; i += kSThreads) {
      sm.hw[i] = 0ull;
      sm.hc[i] = 0u;
    }
    __syncthreads();
    each4(z, V, [&](int v, float zv) {
      if (zv <= hi && zv >= lo && in(v, zv)) {
        const int b = bin_of(zv);
        atomicAdd(&sm.hw[b], weight(v, zv));
      }
    });
    __syncthreads();
    if (warp == 0) {  // the first bin (from the top) where the running weight reaches need
      constexpr int PER = kSBins / 32;
      unsigned long long s = 0;
      for (int i = 0; i < PER; ++i) s += sm.hw[lane * PER + i];
      unsigned long long x = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      unsigned long long nd = need;
      if (nd == 0ull) {  // fraction of the set's weight, all of it in this first histogram
        const unsigned long long w = __shfl_sync(0xFFFFFFFFu, x, 31);
        nd = static_cast<unsigned long long>(ceil(static_cast<double>(frac) * static_cast<double>(w)));
        nd = nd < 1ull ? 1ull : (nd > w ? w : nd);
      }
      const unsigned ball = __ballot_sync(0xFFFFFFFFu, above + x >= nd);
      if (ball == 0u) {  // the finite values hold less than need: the boundary is at -inf
        if (lane == 31) {
          sm.bin = -1;
          sm.above_bin = above + x;
        }
      } else if (lane == __ffs(ball) - 1) {
        unsigned long long acc = above + x - s;
        int b = lane * PER + PER - 1;
        for (int i = 0; i < PER; ++i) {
          const int bb = lane * PER + i;
          if (acc + sm.hw[bb] >= nd) {
            b = bb;
            break;
          }
          acc += sm.hw[bb];
        }
        sm.bin = b;
        sm.above_bin = acc;
      }
      if (lane == 0) sm.need = nd;
    }
    __syncthreads();
    const int B = sm.bin;
    const unsigned long long aB = sm.above_bin;
    need = sm.need;
    __syncthreads();
    if (B < 0) {
      Sel r;
      r.zb = -INFINITY;
      r.ib = first_over(z, V, [&](int v, float zv) { return zv == -INFINITY && in(v, zv) ? weight(v, zv) : 0ull; },
                        need - aB - 1, sm);
      r.wsel = need;
      __syncthreads();
      return r;
    }
    if (t == 0) sm.ncand = 0u;
    __syncthreads();
    each4(z, V, [&](int v, float zv) {  // the bin's tokens, to sort exactly if they fit
      if (zv <= hi && zv >= lo && in(v, zv) && bin_of(zv) == B) {
        const unsigned slot = atomicAdd(&sm.ncand, 1u);
        if (slot < static_cast<unsigned>(kSCand))
          sm.cand[slot] = (static_cast<unsigned long long>(order_key(zv)) << 32) |
                          (0xFFFFFFFFull - static_cast<unsigned>(v));
      }
    });
    __syncthreads();
    const unsigned cB = sm.ncand;
    __syncthreads();
    if (cB <= static_cast<unsigned>(kSCand)) {
      const int n = static_cast<int>(cB);
      int P = 1;
      while (P < n) P <<= 1;
      for (int i = n + t; i < P; i += kSThreads) sm.cand[i] = 0ull;
      if (t == 0) {  // the bin holds at least one token of positive weight; a default all the same
        sm.zb = hi;
        sm.ib = INT_MAX;
        sm.r64 = aB;
      }
      __syncthreads();
      sort_cand(P, true, sm);
      if (warp == 0 && n > 0) {  // the first sorted token at which the running weight reaches need
        const int per = (n + 31) / 32, i0 = min(n, lane * per), i1 = min(n, i0 + per);
        unsigned long long s = 0;
        for (int i = i0; i < i1; ++i) {
          const int v = static_cast<int>(0xFFFFFFFFull - (sm.cand[i] & 0xFFFFFFFFull));
          s += weight(v, z[v]);
        }
        unsigned long long x = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
          if (lane >= o) x += y;
        }
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, aB + x >= need);
        const int L = ball ? __ffs(ball) - 1 : 31;
        if (lane == L) {
          unsigned long long acc = aB + x - s;
          int last = n - 1;
          for (int i = i0; i < i1; ++i) {
            const int v = static_cast<int>(0xFFFFFFFFull - (sm.cand[i] & 0xFFFFFFFFull));
            acc += weight(v, z[v]);
            if (acc >= need) {
              last = i;
              break;
            }
          }
          const int v = static_cast<int>(0xFFFFFFFFull - (sm.cand[last] & 0xFFFFFFFFull));
          sm.zb = z[v];
          sm.ib = v;
          sm.r64 = acc;
        }
      }
      __syncthreads();
      Sel r{sm.zb, sm.ib, sm.r64};
      __syncthreads();
      return r;
    }
    // too many tokens in the bin: zoom into its own range
    float bmax = -INFINITY, bmin = INFINITY;
    each4(z, V, [&](int v, float zv) {
      if (zv <= hi && zv >= lo && in(v, zv) && bin_of(zv) == B) {
        bmax = fmaxf(bmax, zv);
        bmin = fminf(bmin, zv);
      }
    });
    block_maxmin(bmax, bmin, sm);
    above = aB;
    hi = bmax;
    lo = bmin;
  }
  // one value left: its tokens in index order
  const float h = hi;
  Sel r;
  r.zb = h;
  r.ib = first_over(z, V, [&](int v, float zv) { return zv == h && in(v, zv) ? weight(v, zv) : 0ull; },
                    need - above - 1, sm);
  r.wsel = above + sm.r64;
  __syncthreads();
  return r;
}

// top_k <= kSCand: every token at or above the top_k boundary's value bin,
// sorted (z descending, index ascending) into sm.cand[0, n); its first top_k
// entries are the kept set.  A count histogram over [l_min, l_max] (one atomic
// per distinct bin per warp) finds the bin; -1 when the tokens down to that
// bin do not fit (or the finite values hold fewer than top_k tokens).
__device__ int topk_list(const float* z, int V, int k, float hi, float lo_all, SampleSm& sm) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int attempt = 0; attempt < 2; ++attempt) {
    // first the top quarter of the value range (few tokens to bin), else all of it
    const float lo = attempt == 0 ? __fsub_rn(hi, __fmul_rn(__fsub_rn(hi, lo_all), 0.25f)) : lo_all;
    const float inv_w = __fdiv_rn(static_cast<float>(kSBins), __fsub_rn(hi, lo));
    if (!(inv_w > 0.f) || !(inv_w < INFINITY)) return -1;
    auto bin_of = [&](float zv) {  // monotone in zv
      const float q = __fmul_rn(__fsub_rn(hi, zv), inv_w);
      return q >= static_cast<float>(kSBins - 1) ? kSBins - 1 : (q > 0.f ? static_cast<int>(q) : 0);
    };
    for (int i = t; i < kSBins; i += kSThreads) sm.hc[i] = 0u;
    __syncthreads();
    const int n4 = (V + 3) >> 2;
    const float4* z4 = reinterpret_cast<const float4*>(z);
    for (int g0 = t; g0 - lane < n4; g0 += 4 * kSThreads) {  // whole warps take every round
      float4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int g = g0 + u * kSThreads;
        q[u] = g < n4 ? z4[g] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float e4[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int v = 4 * (g0 + u * kSThreads) + e;
          const bool in = v < V && e4[e] >= lo;
          if (__any_sync(0xFFFFFFFFu, in)) {  // one atomic per distinct bin of the warp
            const int b = in ? bin_of(e4[e]) : -1;
            const unsigned m = __match_any_sync(0xFFFFFFFFu, b);
            if (in && lane == __ffs(m) - 1) atomicAdd(&sm.hc[b], static_cast<unsigned>(__popc(m)));
          }
        }
      }
    }
    __syncthreads();
    if (warp == 0) {  // the first bin (from the top) where the running count reaches k
      constexpr int PER = kSBins / 32;
      unsigned s = 0;
      for (int i = 0; i < PER; ++i) s += sm.hc[lane * PER + i];
      unsigned x = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      const unsigned ball = __ballot_sync(0xFFFFFFFFu, x >= static_cast<unsigned>(k));
      if (!ball) {
        if (lane == 0) sm.bin = -2;  // fewer than k tokens in the range
      } else if (lane == __ffs(ball) - 1) {
        unsigned acc = x - s;
        int b = lane * PER + PER - 1;
        for (int i = 0; i < PER; ++i) {
          const int bb = lane * PER + i;
          if (acc + sm.hc[bb] >= static_cast<unsigned>(k)) {
            b = bb;
            break;
          }
          acc += sm.hc[bb];
        }
        sm.bin = acc + sm.hc[b] <= static_cast<unsigned>(kSCand) ? b : -1;
      }
    }
    __syncthreads();
    const int B = sm.bin;
    if (t == 0) sm.ncand = 0u;
    __syncthreads();
    if (B == -2) continue;
    if (B < 0) return -1;
    each4(z, V, [&](int v, float zv) {
      if (zv >= lo && bin_of(zv) <= B) {
        const unsigned slot = atomicAdd(&sm.ncand, 1u);
        if (slot < static_cast<unsigned>(kSCand))
          sm.cand[slot] = (static_cast<unsigned long long>(order_key(zv)) << 32) |
                          (0xFFFFFFFFull - static_cast<unsigned>(v));
      }
    });
    __syncthreads();
    const int n = static_cast<int>(min(sm.ncand, static_cast<unsigned>(kSCand)));
    int P = 1;
    while (P < n) P <<= 1;
    for (int i = n + t; i < P; i += kSThreads) sm.cand[i] = 0ull;
    __syncthreads();
    sort_cand(P, true, sm);
    return n >= k ? n : -1;
  }
  return -1;
}

// top_p, min_p and the draw on the list sm.cand[0, n) sorted (penalised
// logit descending, index ascending), n >= top_k: its first top_k entries are
// the kept set of step 3.  Returns the drawn token (every thread).
__device__ int list_draw(int n, const SampleArgs& a, const LWeight& wl, unsigned long long m24, SampleSm& sm) {
  const float zmax = wl.zmax;
  const int t = threadIdx.x;
  const int K = a.top_k;
  auto w_desc = [&](int i) { return wl(key_float(static_cast<uint32_t>(sm.cand[i] >> 32))); };
  int nk = K;
  if (a.top_p < 1.f) {
    unsigned long long wk = 0;
    for (int i = t; i < K; i += kSThreads) wk += w_desc(i);
    wk = block_sum(wk, sm);
    unsigned long long need =
        static_cast<unsigned long long>(ceil(static_cast<double>(a.top_p) * static_cast<double>(wk)));
    need = need < 1ull ? 1ull : (need > wk ? wk : need);
    nk = list_first_ge(K, w_desc, need, sm) + 1;
  }
  // min_p, then the kept tokens in index order: (index << 32) | key
  int P = 1;
  while (P < n) P <<= 1;
  unsigned long long kept = 0;
  for (int i = t; i < P; i += kSThreads) {
    const unsigned long long c = sm.cand[i];
    bool keep = false;
    if (i < nk) {
      const float lv = key_float(static_cast<uint32_t>(c >> 32));
      keep = __fsub_rn(__fdiv_rn(lv, a.temperature), zmax) >= a.ln_min_p;
    }
    const unsigned long long v = 0xFFFFFFFFull - (c & 0xFFFFFFFFull);
    sm.cand[i] = keep ? ((v << 32) | (c >> 32)) : ~0ull;
    kept += keep ? 1ull : 0ull;
  }
  const int nkept = static_cast<int>(block_sum(kept, sm));
  sort_cand(P, false, sm);
  auto w_idx = [&](int i) { return wl(key_float(static_cast<uint32_t>(sm.cand[i] & 0xFFFFFFFFull))); };
  unsigned long long W = 0;
  for (int i = t; i < nkept; i += kSThreads) W += w_idx(i);
  W = block_sum(W, sm);
  const unsigned long long target = (W >> 24) * m24 + (((W & 0xFFFFFFull) * m24) >> 24);  // floor(u W)
  const int i = list_first_ge(nkept, w_idx, target + 1ull, sm);
  return static_cast<int32_t>(sm.cand[i] >> 32);
}

// The first pass of a top_k <= kSamplePartK draw: block (x, y) takes the
// vocabulary slice [x kSampleSlice, (x + 1) kSampleSlice) of sequence y,
// counts the history tokens that fall in it, applies the penalties exactly as
// k_sample does (step 1), and writes the slice's first top_k entries in the
// order of step 2 as keys (order key of l << 32 | 2^32 - 1 - index) to
// DevSeq::sparts.  Every token of the global first top_k is among its
// slice's first top_k, so the merge needs nothing else.
constexpr int kPThreads = 256;
__global__ void __launch_bounds__(kPThreads) k_sample_part(const DevSeq* seqs, int V, int max_seq, SampleArgs a) {
  __shared__ unsigned long long key[kSampleSlice];
  __shared__ unsigned int cnt[kSampleSlice];
  const DevSeq& s = seqs[blockIdx.y];
  const int t = threadIdx.x;
  const uint32_t S = s.state->pos;
  if (S == 0u || S > static_cast<uint32_t>(max_seq)) return;
  const int v0 = static_cast<int>(blockIdx.x) * kSampleSlice;
  if (a.penalize) {
    for (int i = t; i < kSampleSlice; i += kPThreads) cnt[i] = 0u;
    __syncthreads();
    for (int i = t; i < static_cast<int>(S); i += kPThreads) {
      const int x = s.tokens[i] - v0;
      if (x >= 0 && x < kSampleSlice) atomicAdd(&cnt[x], 1u);
    }
    __syncthreads();
  }
  for (int i = t; i < kSampleSlice; i += kPThreads) {
    const int v = v0 + i;
    unsigned long long k = 0ull;  // below every token's key: the slice's padding
    if (v < V) {
      float l = s.logits[v];
      if (isnan(l)) l = -INFINITY;
      const unsigned c = a.penalize ? cnt[i] : 0u;
      if (c && l > -INFINITY) {
        l = l > 0.f ? __fdiv_rn(l, a.repeat) : __fmul_rn(l, a.repeat);
        l = __fsub_rn(l, a.presence);
        l = __fsub_rn(l, __fmul_rn(a.frequency, static_cast<float>(c)));
        if (isnan(l)) l = -INFINITY;
      }
      k = (static_cast<unsigned long long>(order_key(l)) << 32) | (0xFFFFFFFFull - static_cast<unsigned>(v));
    }
    key[i] = k;
  }
  __syncthreads();
  for (int k2 = 2; k2 <= kSampleSlice; k2 <<= 1)  // bitonic sort, descending
    for (int j = k2 >> 1; j > 0; j >>= 1) {
      for (int i = t; i < kSampleSlice; i += kPThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long x = key[i], y = key[ixj];
          if (((i & k2) == 0) ? (x < y) : (x > y)) {
            key[i] = y;
            key[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  unsigned long long* out = s.sparts + static_cast<size_t>(blockIdx.x) * kSamplePartK;
  for (int i = t; i < a.top_k; i += kPThreads) out[i] = key[i];
}

__global__ void __launch_bounds__(kSThreads, 1) k_sample(const DevSeq* seqs, int V, int max_seq, SampleArgs a) {
  __shared__ SampleSm sm;
  const DevSeq& s = seqs[blockIdx.x];
  const int t = threadIdx.x;
  const uint32_t S = s.state->pos;  // inputs so far; the drawn token becomes the input at S
  if (S == 0u || S > static_cast<uint32_t>(max_seq)) return;
  const float* lg = s.logits;
  float* z = s.sz;
  uint32_t* cnt = s.scnt;
  int32_t* tok = s.tokens;
  const int n_in = static_cast<int>(S);
  if (!(a.temperature > 0.f)) {  // the greedy token of the raw logits: ties to the lower index, NaN never wins
    float bv = -INFINITY;
    int bi = INT_MAX;
    each4(lg, V, [&](int v, float l) {
      if (!isnan(l) && (l > bv || (l == bv && v < bi))) {
        bv = l;
        bi = v;
      }
    });
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((t & 31) == 0) {
      sm.fa[t >> 5] = bv;
      sm.cand[t >> 5] = static_cast<unsigned long long>(static_cast<unsigned>(bi));
    }
    __syncthreads();
    if (t == 0) {
      for (int w = 1; w < kSWarps; ++w) {
        const float ov = sm.fa[w];
        const int oi = static_cast<int>(sm.cand[w]);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (bi == INT_MAX) {
        atomicOr(&s.state->err, kErrAllNaN);
        bi = -1;
      }
      tok[S] = bi;
    }
    return;
  }
  if (a.parts > 0) {
    // the slices' first top_k entries hold the global first top_k.  tau, the
    // top_k-th largest of the slices' first m keys (a subset of those
    // entries), is at most the global top_k-th key, so the keys at or above
    // tau hold the first top_k; with m large enough for the subset to hold
    // top_k keys, few more than top_k survive unless one slice holds most of
    // them
    const int K = a.top_k, np = a.parts;
    const unsigned long long* sp = s.sparts;
    int m = (2 * K + np - 1) / np;
    m = m < 4 ? 4 : m;
    m = m > K ? K : m;
    if (np * m > kSCand) m = kSCand / np;
    const int ns = np * m;
    int Ps = 1;
    while (Ps < ns) Ps <<= 1;
    for (int i = t; i < Ps; i += kSThreads) {
      unsigned long long k = 0ull;
      if (i < ns) {
        const int b = i / m, j = i - b * m;
        k = __ldcg(sp + static_cast<size_t>(b) * kSamplePartK + j);
      }
      sm.cand[i] = k;
    }
    if (t == 0) sm.ncand = 0u;
    __syncthreads();
    sort_cand(Ps, true, sm);
    const unsigned long long tau = ns >= K ? sm.cand[K - 1] : 0ull;
    __syncthreads();
    for (int i = t; i < np * K; i += kSThreads) {
      const int b = i / K, j = i - b * K;
      const unsigned long long k = __ldcg(sp + static_cast<size_t>(b) * kSamplePartK + j);
      if (k >= tau) {
        const unsigned slot = atomicAdd(&sm.ncand, 1u);
        if (slot < static_cast<unsigned>(kSCand)) sm.cand[slot] = k;
      }
    }
    __syncthreads();
    const unsigned nc = sm.ncand;
    if (nc <= static_cast<unsigned>(kSCand)) {
      const int n = static_cast<int>(nc);
      int P = 1;
      while (P < n) P <<= 1;
      for (int i = n + t; i < P; i += kSThreads) sm.cand[i] = 0ull;
      __syncthreads();
      sort_cand(P, true, sm);
      const float lmax = key_float(static_cast<uint32_t>(sm.cand[0] >> 32));
      const float zmax = __fdiv_rn(lmax, a.temperature);
      // every logit NaN, or l_max / T overflowing: the one-pass path below decides
      if (n >= K && lmax > -INFINITY && zmax > -INFINITY && zmax < INFINITY) {
        const LWeight wl{a.temperature, zmax};
        const unsigned long long m24 = mix64(a.seed + (static_cast<unsigned long long>(S) + 1ull) * kGolden) >> 40;
        const int v = list_draw(n, a, wl, m24, sm);
        if (t == 0) tok[S] = v;
        return;
      }
    }
    __syncthreads();
  }
  if (a.penalize)
    for (int i = t; i < n_in; i += kSThreads) {
      const int x = tok[i];
      if (x >= 0 && x < V) atomicAdd(&cnt[x], 1u);
    }
  // the penalised logits, four float4 groups in flight per thread; the counts
  // are read beside the logits and zeroed; the padding gets -inf
  __syncthreads();
  float lmax = -INFINITY, lmin = INFINITY;
  {
    const int n4 = (V + 3) >> 2;
    const float4* l4 = reinterpret_cast<const float4*>(lg);
    float4* z4 = reinterpret_cast<float4*>(z);
    uint4* c4 = reinterpret_cast<uint4*>(cnt);
    auto tz = [&](float l, unsigned c, int v) {
      if (v >= V || isnan(l)) return -INFINITY;
      if (c) {
        l = l > 0.f ? __fdiv_rn(l, a.repeat) : __fmul_rn(l, a.repeat);
        l = __fsub_rn(l, a.presence);
        l = __fsub_rn(l, __fmul_rn(a.frequency, static_cast<float>(c)));
        if (isnan(l)) return -INFINITY;
      }
      lmax = fmaxf(lmax, l);
      if (l > -INFINITY) lmin = fminf(lmin, l);
      return l;
    };
    for (int g0 = t; g0 < n4; g0 += 4 * kSThreads) {
      float4 q[4];
      uint4 cc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int g = g0 + u * kSThreads;
        q[u] = g < n4 ? l4[g] : make_float4(0.f, 0.f, 0.f, 0.f);
        cc[u] = g < n4 && a.penalize ? c4[g] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int g = g0 + u * kSThreads;
        if (g < n4) {
          const int v = 4 * g;
          z4[g] = make_float4(tz(q[u].x, cc[u].x, v), tz(q[u].y, cc[u].y, v + 1), tz(q[u].z, cc[u].z, v + 2),
                              tz(q[u].w, cc[u].w, v + 3));
          if (cc[u].x | cc[u].y | cc[u].z | cc[u].w) c4[g] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
  }
  block_maxmin(lmax, lmin, sm);
  if (!(lmax > -INFINITY)) {  // every logit NaN
    if (t == 0) {
      atomicOr(&s.state->err, kErrAllNaN);
      tok[S] = -1;
    }
    return;
  }
  const float zmax = __fdiv_rn(lmax, a.temperature);
  if (!(zmax > -INFINITY && zmax < INFINITY)) {  // l_max / T overflows: the T -> 0 limit, greedy on l
    const float lm = lmax;
    const int v = first_over(z, V, [lm](int, float lv) { return lv == lm ? 1ull : 0ull; }, 0ull, sm);
    if (t == 0) tok[S] = v;
    return;
  }
  const LWeight wl{a.temperature, zmax};
  const unsigned long long m24 = mix64(a.seed + (static_cast<unsigned long long>(S) + 1ull) * kGolden) >> 40;
  Keep kp{-INFINITY, INT_MAX, -INFINITY, INT_MAX, a.temperature, zmax, a.ln_min_p};
  if (a.top_k >= 1 && a.top_k < V && a.top_k <= kSCand) {
    // the kept tokens fit shared memory: top_p, min_p and the draw on that list
    const int n = topk_list(z, V, a.top_k, lmax, lmin, sm);
    if (n >= 0) {
      const int v = list_draw(n, a, wl, m24, sm);
      if (t == 0) tok[S] = v;
      return;
    }
  }
  if (a.top_k >= 1 && a.top_k < V) {
    const Sel r = select_top(
        z, V, [](int, float) { return true; }, [](int, float) { return 1ull; },
        static_cast<unsigned long long>(a.top_k), 0.f, lmax, lmin, sm);
    kp.kz = r.zb;
    kp.ki = r.ib;
  }
  unsigned long long W = 0;
  bool have_w = false;
  if (a.top_p < 1.f) {
    const float kz = kp.kz;
    const int ki = kp.ki;
    const Sel r = select_top(
        z, V, [kz, ki](int v, float zv) { return zv > kz || (zv == kz && v <= ki); },
        [wl](int, float lv) { return wl(lv); }, 0ull, a.top_p, lmax, fmaxf(lmin, kz), sm);
    kp.pz = r.zb;
    kp.pi = r.ib;
    W = r.wsel;  // the kept mass, unless min_p removes more
    have_w = !(a.ln_min_p > -INFINITY);
  }
  if (!have_w) {
    W = 0;
    each4(z, V, [&](int v, float zv) {
      if (kp(v, zv)) W += wl(zv);
    });
    W = block_sum(W, sm);
  }
  // the draw
  const unsigned long long target = (W >> 24) * m24 + (((W & 0xFFFFFFull) * m24) >> 24);  // floor(u W)
  const int v = first_over(
      z, V, [&](int i, float zv) { return kp(i, zv) ? wl(zv) : 0ull; }, target, sm);
  if (t == 0) tok[S] = v < V ? v : V - 1;
}

}  // namespace

cudaError_t launch_sample(const DevSeq* seqs, int n, int V, int max_seq, const SampleArgs& a, cudaStream_t st,
                          bool slices) {
  SampleArgs b = a;
  b.parts = 0;
  if (slices && a.temperature > 0.f && a.top_k >= 1 && a.top_k <= kSamplePartK && a.top_k < V) {
    b.parts = (V + kSampleSlice - 1) / kSampleSlice;
    k_sample_part<<<dim3(b.parts, n), kPThreads, 0, st>>>(seqs, V, max_seq, b);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  k_sample<<<n, kSThreads, 0, st>>>(seqs, V, max_seq, b);
  return cudaGetLastError();
}

}  // namespace tqd
