// Seeded sampling of the next token from a step's logits ("Metal LLM decode",
// the sampled arm of the batched prefill+decode section: temperature, top_k,
// top_p, min_p, repeat / presence / frequency penalties and a seed;
// temperature <= 0 falls back to the greedy token and top_k = 1 reproduces
// it).  One block per sequence, in this order:
//   1. penalties on the distinct tokens among the sequence's inputs (counted
//      in a per-sequence array the block leaves zeroed), each an f32
//      operation: a = l > 0 ? l / r : l * r; a -= presence; a -= frequency * c;
//   2. z = l / T in f32 (NaN -> -inf), into a per-sequence array;
//   3. top_k: the k largest z, ties to the lower index;
//   4. top_p: of those, in the order (z descending, index ascending), the
//      shortest prefix whose mass reaches p of their mass;
//   5. min_p: z - z_max >= ln(min_p) (f32 difference; the log taken on the host);
//   6. draw: u = the top 24 bits of splitmix64's output at the drawn token's
//      position, times 2^-24; the token is the first kept one in index order
//      whose running mass exceeds u times the kept mass.
// Masses are exp(z - z_max) in f32, carried as integers in units of 2^-32 of
// the most likely token's, so every sum is exact and independent of order and
// the draw is deterministic.  A boundary (steps 3, 4) is found by a histogram
// of the values over [z_min, z_max], then an exact sort of the boundary bin's
// tokens (a zoom into the bin when it holds too many), ties in index order.
#include <climits>

#include "tqd_internal.h"

namespace tqd {
namespace {

constexpr int kSThreads = 512;
constexpr int kSWarps = kSThreads / 32;
constexpr int kSBins = 2048;                // value bins of a boundary search
constexpr int kSCand = 2048;                // tokens of a boundary bin sorted exactly
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
  unsigned long long above_bin;
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

// A token v of value z is kept when it passes every stage set so far.
struct Keep {
  float kz;
  int ki;      // top_k: z > kz, or z == kz and v <= ki
  float pz;
  int pi;      // top_p: the same
  float zmax;
  float lnmp;  // min_p: z - zmax >= lnmp (-inf when off)
  __device__ bool operator()(int v, float z) const {
    return (z > kz || (z == kz && v <= ki)) && (z > pz || (z == pz && v <= pi)) && __fsub_rn(z, zmax) >= lnmp;
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

// The smallest v < V whose running weight (over 0..v, index order) exceeds
// thresh; V when the total does not.
template <class Wt>
__device__ int first_over(const float* z, int V, Wt weight, unsigned long long thresh, SampleSm& sm) {
  constexpr int E = 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long run = 0;
  for (int base = 0; base < V; base += kSThreads * E) {
    const int v0 = base + static_cast<int>(threadIdx.x) * E;
    unsigned long long w[E], s = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      w[e] = v0 + e < V ? weight(v0 + e, z[v0 + e]) : 0ull;
      s += w[e];
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
#pragma unroll
        for (int e = 0; e < E; ++e) {
          acc += w[e];
          if (acc > thresh) {
            sm.ib = v0 + e;
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

// The boundary (zb, ib) of the first `need` weight units of the tokens that
// pass `in`, in the order (z descending, index ascending): those tokens are
// exactly the ones passing `in` with z > zb, or z == zb and index <= ib.
// hi: the set's largest value; lo: a lower bound of its finite values;
// 1 <= need <= the set's weight.
template <class In, class Wt>
__device__ void select_top(const float* z, int V, In in, Wt weight, unsigned long long need, float hi, float lo,
                           SampleSm& sm, float& zb, int& ib) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  unsigned long long above = 0;  // weight of the set's tokens above hi
  for (int round = 0; round < 8 && hi > lo; ++round) {
    const float width = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(kSBins));
    if (!(width > 0.f)) break;
    auto bin_of = [&](float zv) {
      const float q = __fdiv_rn(__fsub_rn(hi, zv), width);
      return q >= static_cast<float>(kSBins - 1) ? kSBins - 1 : (q > 0.f ? static_cast<int>(q) : 0);
    };
    for (int i = t; i < kSBins; i += kSThreads) {
      sm.hw[i] = 0ull;
      sm.hc[i] = 0u;
    }
    __syncthreads();
    for (int v = t; v < V; v += kSThreads) {
      const float zv = z[v];
      if (zv <= hi && zv >= lo && in(v, zv)) {
        const int b = bin_of(zv);
        atomicAdd(&sm.hw[b], weight(v, zv));
        atomicAdd(&sm.hc[b], 1u);
      }
    }
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
      const unsigned ball = __ballot_sync(0xFFFFFFFFu, above + x >= need);
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
          if (acc + sm.hw[bb] >= need) {
            b = bb;
            break;
          }
          acc += sm.hw[bb];
        }
        sm.bin = b;
        sm.above_bin = acc;
        sm.cnt_bin = sm.hc[b];
      }
    }
    __syncthreads();
    const int B = sm.bin;
    const unsigned long long aB = sm.above_bin;
    const unsigned int cB = sm.cnt_bin;
    __syncthreads();
    if (B < 0) {
      zb = -INFINITY;
      ib = first_over(z, V, [&](int v, float zv) { return zv == -INFINITY && in(v, zv) ? weight(v, zv) : 0ull; },
                      need - aB - 1, sm);
      return;
    }
    if (cB <= static_cast<unsigned>(kSCand)) {  // sort the bin's tokens exactly
      if (t == 0) sm.ncand = 0u;
      __syncthreads();
      for (int v = t; v < V; v += kSThreads) {
        const float zv = z[v];
        if (zv <= hi && zv >= lo && in(v, zv) && bin_of(zv) == B) {
          const unsigned slot = atomicAdd(&sm.ncand, 1u);
          if (slot < static_cast<unsigned>(kSCand))
            sm.cand[slot] = (static_cast<unsigned long long>(order_key(zv)) << 32) |
                            (0xFFFFFFFFull - static_cast<unsigned>(v));
        }
      }
      __syncthreads();
      const int n = static_cast<int>(min(sm.ncand, static_cast<unsigned>(kSCand)));
      int P = 1;
      while (P < n) P <<= 1;
      for (int i = n + t; i < P; i += kSThreads) sm.cand[i] = 0ull;
      __syncthreads();
      for (int k = 2; k <= P; k <<= 1)  // bitonic sort, descending
        for (int j = k >> 1; j > 0; j >>= 1) {
          for (int i = t; i < P; i += kSThreads) {
            const int ixj = i ^ j;
            if (ixj > i) {
              const unsigned long long a = sm.cand[i], b = sm.cand[ixj];
              if (((i & k) == 0) ? (a < b) : (a > b)) {
                sm.cand[i] = b;
                sm.cand[ixj] = a;
              }
            }
          }
          __syncthreads();
        }
      if (t == 0) {  // the bin holds at least one token of positive weight; a default all the same
        sm.zb = hi;
        sm.ib = INT_MAX;
      }
      __syncthreads();
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
        }
      }
      __syncthreads();
      zb = sm.zb;
      ib = sm.ib;
      __syncthreads();
      return;
    }
    // too many tokens in the bin: zoom into its own range
    float bmax = -INFINITY, bmin = INFINITY;
    for (int v = t; v < V; v += kSThreads) {
      const float zv = z[v];
      if (zv <= hi && zv >= lo && in(v, zv) && bin_of(zv) == B) {
        bmax = fmaxf(bmax, zv);
        bmin = fminf(bmin, zv);
      }
    }
    block_maxmin(bmax, bmin, sm);
    above = aB;
    hi = bmax;
    lo = bmin;
  }
  // one value left: its tokens in index order
  const float h = hi;
  zb = h;
  ib = first_over(z, V, [&](int v, float zv) { return zv == h && in(v, zv) ? weight(v, zv) : 0ull; },
                  need - above - 1, sm);
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
  if (a.penalize)
    for (int i = t; i < n_in; i += kSThreads) {
      const int x = tok[i];
      if (x >= 0 && x < V) atomicAdd(&cnt[x], 1u);
    }
  for (int v = t; v < V; v += kSThreads) {
    const float l = lg[v];
    z[v] = isnan(l) ? -INFINITY : __fdiv_rn(l, a.temperature);
  }
  __syncthreads();
  if (a.penalize) {
    for (int i = t; i < n_in; i += kSThreads) {
      const int x = tok[i];
      if (x < 0 || x >= V) continue;
      const unsigned c = atomicExch(&cnt[x], 0u);  // one thread per distinct token
      if (c == 0u) continue;
      float l = lg[x];
      if (isnan(l)) continue;
      l = l > 0.f ? __fdiv_rn(l, a.repeat) : __fmul_rn(l, a.repeat);
      l = __fsub_rn(l, a.presence);
      l = __fsub_rn(l, __fmul_rn(a.frequency, static_cast<float>(c)));
      z[x] = isnan(l) ? -INFINITY : __fdiv_rn(l, a.temperature);
    }
  }
  __syncthreads();
  float zmax = -INFINITY, zmin = INFINITY;
  for (int v = t; v < V; v += kSThreads) {
    const float zv = z[v];
    zmax = fmaxf(zmax, zv);
    if (zv > -INFINITY) zmin = fminf(zmin, zv);
  }
  block_maxmin(zmax, zmin, sm);
  if (!(zmax > -INFINITY) || !(zmax < INFINITY)) {  // every logit NaN, or z overflowed
    if (t == 0) {
      atomicOr(&s.state->err, kErrAllNaN);
      tok[S] = -1;
    }
    return;
  }
  Keep kp{-INFINITY, INT_MAX, -INFINITY, INT_MAX, zmax, a.ln_min_p};
  if (a.top_k >= 1 && a.top_k < V) {
    float zb;
    int ib;
    select_top(
        z, V, [](int, float) { return true; }, [](int, float) { return 1ull; },
        static_cast<unsigned long long>(a.top_k), zmax, zmin, sm, zb, ib);
    kp.kz = zb;
    kp.ki = ib;
  }
  if (a.top_p < 1.f) {
    const float kz = kp.kz;
    const int ki = kp.ki;
    auto in_k = [kz, ki](int v, float zv) { return zv > kz || (zv == kz && v <= ki); };
    auto wt = [zmax](int, float zv) { return wfix(zv, zmax); };
    unsigned long long wk = 0;
    for (int v = t; v < V; v += kSThreads) {
      const float zv = z[v];
      if (in_k(v, zv)) wk += wt(v, zv);
    }
    wk = block_sum(wk, sm);
    unsigned long long need =
        static_cast<unsigned long long>(ceil(static_cast<double>(a.top_p) * static_cast<double>(wk)));
    if (need < 1ull) need = 1ull;
    if (need > wk) need = wk;
    float zb;
    int ib;
    select_top(z, V, in_k, wt, need, zmax, fmaxf(zmin, kz), sm, zb, ib);
    kp.pz = zb;
    kp.pi = ib;
  }
  // the draw
  unsigned long long W = 0;
  for (int v = t; v < V; v += kSThreads) {
    const float zv = z[v];
    if (kp(v, zv)) W += wfix(zv, zmax);
  }
  W = block_sum(W, sm);
  const unsigned long long m24 = mix64(a.seed + (static_cast<unsigned long long>(S) + 1ull) * kGolden) >> 40;
  const unsigned long long target = (W >> 24) * m24 + (((W & 0xFFFFFFull) * m24) >> 24);  // floor(u W)
  const int v = first_over(
      z, V, [&](int i, float zv) { return kp(i, zv) ? wfix(zv, zmax) : 0ull; }, target, sm);
  if (t == 0) tok[S] = v < V ? v : V - 1;
}

}  // namespace

cudaError_t launch_sample(const DevSeq* seqs, int n, int V, int max_seq, const SampleArgs& a, cudaStream_t st) {
  k_sample<<<n, kSThreads, 0, st>>>(seqs, V, max_seq, a);
  return cudaGetLastError();
}

}  // namespace tqd
