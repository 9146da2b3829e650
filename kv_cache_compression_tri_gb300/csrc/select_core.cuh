// select_core.cuh -- per-slice budgeted selection, one CTA per slice
// (the kernels and key sources; select.cu launches them, select_compact.cu
// fuses the selection with the compaction).
//
// Keep [0, P) U top-(B-P-W) candidates U [n-W, n), ascending; among equal
// keys the lower slot wins. Three key sources share the kernel (the third,
// ZMaxKeys, ranks by the GQA z-score maximum, below):
//   * scores -- TriAttention paper summary, "Retention and eviction" (top-B
//     by score); Random Attention, Eq. 2 (top-K with the prompt forced in):
//     the key of candidate i is the order-preserving u32 of its fp32 score;
//   * uniform draws -- Random Attention, section 3 (Eq. 3, Algorithm 1): the
//     key of candidate i is word (i mod 4) of Philox-4x32-10 with counter
//     (i/4, head + 65536 layer, seq, round) and key = the seed; the recent
//     buffer is kept unscored (section 2).
//
// Nothing is staged; a slice costs one streaming pass over its keys:
//   1. a window [t_lo, t_hi] that holds the need-th largest key with high
//      probability. Draws: the need-th largest of m i.i.d. uniforms has mean
//      1 - need/(m+1) and variance need (m+1-need) / ((m+1)^2 (m+2)); the
//      window is +-8 standard deviations. Scores: a systematic sample of 2048
//      candidates; the sample keys of rank r* -+ 4.5 sd (r* = need 2048 / m)
//      are found by a radix select on the sample and bound the window. A
//      slice with at most LCAP candidates takes the whole key range;
//   2. the pass: keys above the window set their slot's bit in an "above"
//      bitmap and are counted; keys inside it join a short list (key, slot);
//   3. if the threshold provably lies in the window (count above < need <=
//      count above + list size, list not overflowed) a radix select on the
//      list alone finds it exactly; otherwise an exact radix select over all
//      candidates (keys re-read or regenerated for every pass) does;
//   4. emission from the "above" and "equal" bitmaps in slot order
//      (per-thread popcounts and one block scan), equal keys ranked by slot,
//      so the keep list comes out ascending without a sort.
// Shared memory stays small (42 KB), so five CTAs share an SM and the
// latency-bound phases of one slice overlap the streaming pass of another.
// Slices whose candidates span more slots than the bitmaps cover rebuild
// the bitmaps piece by piece for the emission.
#pragma once

#include <cuda_runtime.h>

#include <math.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

constexpr int NT = 256;              // threads per CTA
constexpr int NW = NT / 32;          // warps
constexpr int MINB = 5;              // CTAs per SM
constexpr int BM_SLOTS = 32768;      // slots covered by one pair of bitmaps
constexpr int BM_WORDS = BM_SLOTS / 32;
constexpr int LCAP = 4096;           // short-list capacity
constexpr int SPT = 8;               // sampled scores per thread
constexpr int NSAMPLE = NT * SPT;    // 2048
constexpr float SAMPLE_SD = 4.5f;    // half-width of the sampled window, in sd
constexpr double DRAW_SD = 8.0;      // half-width of the uniform-draw window, in sd

struct SSmem {
  uint32_t gt[BM_WORDS];  // slot above the threshold
  uint32_t eq[BM_WORDS];  // slot equal to the threshold (candidate tie)
  uint32_t lkey[LCAP];
  int32_t lslot[LCAP];
  unsigned hist[2][256];
  unsigned wsum[NW];
  uint32_t wmin[NW], wmax[NW];
  int pick_digit[2];
  unsigned pick_above[2], pick_count[2];
  unsigned nlist, cnt_hi, total;
  uint32_t t_lo, t_hi;
  int nan_seen;
};

struct Ctx {
  int64_t s;
  int n, P, W, B;
  int lo;   // first slot of the swept range (P rounded down to 4)
  int end;  // n - W: exclusive end of the candidates
};

__device__ __forceinline__ bool in_range(int i, int lo, int hi) {
  return static_cast<unsigned>(i - lo) < static_cast<unsigned>(hi - lo);
}

// Bits e of slots i0 + e (e < 4) that lie in [lo, hi).
__device__ __forceinline__ uint32_t valid_bits(int i0, int lo, int hi) {
  if (i0 >= lo && i0 + 3 < hi) return 0xfu;
  uint32_t v = 0u;
#pragma unroll
  for (int e = 0; e < 4; ++e) v |= static_cast<uint32_t>(in_range(i0 + e, lo, hi)) << e;
  return v;
}

// digit b with count(digits > b) < need <= count(digits >= b) in h[256],
// by one warp; published in slot `which` of the pick fields.
__device__ __forceinline__ void pick_bin(SSmem& sm, const unsigned* hist, unsigned need, int lane, int which) {
  unsigned h[8], ls = 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = hist[lane * 8 + j];
    ls += h[j];
  }
  unsigned suf = ls;  // inclusive suffix sum over lanes >= this lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_down_sync(FULL_MASK, suf, o);
    if (lane + o < 32) suf += y;
  }
  const unsigned above_lane = suf - ls;
  if (above_lane < need && need <= suf) {
    unsigned cum = above_lane;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      if (cum + h[j] >= need) {
        sm.pick_digit[which] = lane * 8 + j;
        sm.pick_above[which] = cum;
        sm.pick_count[which] = h[j];
        break;
      }
      cum += h[j];
    }
  }
}

// State of one radix select: keys matching (prefix, mask) are still in
// play; the next digit is `width` bits at `shift`; `need` counts from the top.
struct Radix {
  uint32_t prefix, mask;
  unsigned need;
  int shift, width;
  bool done;

  // Start below the bits that every key in [kmin, kmax] shares.
  __device__ __forceinline__ void start(uint32_t kmin, uint32_t kmax, unsigned need_) {
    need = need_;
    const uint32_t diff = kmin ^ kmax;
    if (diff == 0u) {  // a single key value: it is the answer
      prefix = kmin;
      mask = 0xffffffffu;
      shift = 0;
      width = 0;
      done = true;
      return;
    }
    const int hb = 31 - __clz(diff);
    shift = max(hb - 7, 0);
    width = hb - shift + 1;
    mask = (hb == 31) ? 0u : ~((2u << hb) - 1u);
    prefix = kmin & mask;
    done = false;
  }
  __device__ __forceinline__ bool matches(uint32_t k) const { return (k & mask) == prefix; }
  __device__ __forceinline__ uint32_t digit(uint32_t k) const { return (k >> shift) & ((1u << width) - 1u); }
  // Take the picked bin; returns its count. Callers decide when to stop.
  __device__ __forceinline__ unsigned take(const SSmem& sm, int which) {
    need -= sm.pick_above[which];
    prefix |= static_cast<uint32_t>(sm.pick_digit[which]) << shift;
    mask |= ((1u << width) - 1u) << shift;
    return sm.pick_count[which];
  }
  __device__ __forceinline__ void next_digit() {
    width = min(8, shift);
    shift -= width;
  }
};

// Block-wide exclusive scan of one value per thread; returns the thread's
// offset, and the total in *total.
__device__ __forceinline__ unsigned block_scan(SSmem& sm, unsigned v, unsigned* total) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  unsigned incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    const unsigned x = (lane < NW) ? sm.wsum[lane] : 0u;
    unsigned xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(FULL_MASK, xi, o);
      if (lane >= o) xi += y;
    }
    if (lane < NW) sm.wsum[lane] = xi - x;
    if (lane == 31) sm.total = xi;
  }
  __syncthreads();
  const unsigned off = incl - v + sm.wsum[w];
  *total = sm.total;
  __syncthreads();
  return off;
}

// Block-wide min and max; every thread gets the result.
__device__ __forceinline__ void block_minmax(SSmem& sm, uint32_t& kmin, uint32_t& kmax) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(FULL_MASK, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(FULL_MASK, kmax, o));
  }
  if (lane == 0) {
    sm.wmin[w] = kmin;
    sm.wmax[w] = kmax;
  }
  __syncthreads();
  kmin = (lane < NW) ? sm.wmin[lane] : 0xffffffffu;
  kmax = (lane < NW) ? sm.wmax[lane] : 0u;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(FULL_MASK, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(FULL_MASK, kmax, o));
  }
  __syncthreads();  // wmin / wmax may be rewritten by the next call
}

// The keys of RUN consecutive slots.
template <int RUN>
struct RunKeys {
  uint32_t k[RUN];
};

// Window from a systematic sample of NSAMPLE candidates spread evenly over
// [P, n - W), taken as NSAMPLE / RUN runs of RUN consecutive slots (each run
// RUN-aligned). Sources that read one score row use RUN = 1; sources that
// read several rows per slot use RUN = 8, one 32-byte sector per row, so the
// sample touches an eighth of the sectors (their CTAs' rows do not stay in L2
// until the pass re-reads them). run_of(s0) gives the keys of slots s0 ..
// s0 + RUN - 1. The sample keys of ranks r* -+ SAMPLE_SD sd bound [t_lo,
// t_hi] (r* = need NSAMPLE / m, sd its binomial standard deviation). Requires
// m > LCAP (>= 2 NSAMPLE slots).
template <int RUN, class RunOf>
__device__ void sampled_window(SSmem& sm, const Ctx& c, int need, int m, const RunOf& run_of, uint32_t& t_lo,
                               uint32_t& t_hi) {
  static_assert(SPT % RUN == 0, "runs per thread");
  constexpr int NRUN = NSAMPLE / RUN;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  uint32_t sk[SPT];
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  const int first = (c.P + RUN - 1) / RUN;  // first RUN-aligned run inside the candidates
  const int last = (c.end - RUN) / RUN;     // last one
#pragma unroll
  for (int q = 0; q < SPT / RUN; ++q) {
    const int j = t + NT * q;  // run index
    const int run = first + static_cast<int>((static_cast<int64_t>(last - first) * j) / (NRUN - 1));
    const RunKeys<RUN> rk = run_of(run * RUN);
#pragma unroll
    for (int r = 0; r < RUN; ++r) {
      sk[q * RUN + r] = rk.k[r];
      kmin = min(kmin, sk[q * RUN + r]);
      kmax = max(kmax, sk[q * RUN + r]);
    }
  }
  block_minmax(sm, kmin, kmax);
  // sample ranks (1 = largest) that bracket the need-th largest candidate
  // (fp32: the window only has to be about right, and the fp64 pipe is slow)
  const float rho = static_cast<float>(need) / static_cast<float>(m);
  const float rs = rho * NSAMPLE, sd = sqrtf(NSAMPLE * rho * (1.0f - rho));
  const int ra = static_cast<int>(floorf(rs - SAMPLE_SD * sd - 1.0f));
  const int rb = static_cast<int>(ceilf(rs + SAMPLE_SD * sd + 1.0f));
  Radix A, B;
  const bool want_a = ra >= 1, want_b = rb <= NSAMPLE;
  A.start(kmin, kmax, static_cast<unsigned>(max(ra, 1)));
  B.start(kmin, kmax, static_cast<unsigned>(min(rb, NSAMPLE)));
  A.done |= !want_a;
  B.done |= !want_b;
  // Refine both ranks together until their bins hold at most 4 sample
  // keys (or the full key is known): t_hi is the top of A's bin, so fewer
  // than ra sample keys lie above it; t_lo the bottom of B's bin, so at
  // least rb lie at or above it.
  while (!(A.done && B.done)) {
    sm.hist[0][t] = 0u;
    sm.hist[1][t] = 0u;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < SPT; ++r) {
      if (!A.done && A.matches(sk[r])) atomicAdd(&sm.hist[0][A.digit(sk[r])], 1u);
      if (!B.done && B.matches(sk[r])) atomicAdd(&sm.hist[1][B.digit(sk[r])], 1u);
    }
    __syncthreads();
    if (w == 0 && !A.done) pick_bin(sm, sm.hist[0], A.need, lane, 0);
    if (w == 1 && !B.done) pick_bin(sm, sm.hist[1], B.need, lane, 1);
    __syncthreads();
    if (!A.done) {
      const unsigned cnt = A.take(sm, 0);
      if (cnt <= 4u || A.shift == 0) A.done = true; else A.next_digit();
    }
    if (!B.done) {
      const unsigned cnt = B.take(sm, 1);
      if (cnt <= 4u || B.shift == 0) B.done = true; else B.next_digit();
    }
  }
  t_hi = want_a ? (A.prefix | ((1u << A.shift) - 1u) | ~A.mask) : 0xffffffffu;
  t_lo = want_b ? (B.prefix & B.mask) : 0u;
}

// ---- key sources --------------------------------------------------------------

// fp32 scores [S][n_cap]; keys of slots outside [P, end) read as 0.
struct ScoreKeys {
  static constexpr int U = 4;  // 16-byte loads in flight per thread
  static constexpr bool GROUPED = false;
  static constexpr bool INTERIOR = true;  // fetch_interior() for groups inside [P, end)
  static constexpr bool PREFETCH = true;  // prefetch() the candidates' scores into L2
  const float* row;
  bool vec;  // 16-byte loads allowed

  __device__ static ScoreKeys make(const SelectParams& p, const Ctx& c, int, int, int) {
    ScoreKeys k;
    k.row = p.scores + c.s * static_cast<int64_t>(p.n_cap);
    k.vec = (reinterpret_cast<uintptr_t>(k.row) & 15) == 0;  // lo is a multiple of 4
    return k;
  }
  // Keys of four slots that all lie in [P, end): one 16-byte load (the row
  // is 16-byte aligned and i0 a multiple of 4 from it) and the key of each
  // score in integer operations, equal to score_key's (NaN -> 0 and flagged,
  // -0 -> +0, then the order-preserving flip).
  __device__ __forceinline__ uint4 fetch_interior(int i0, bool& nan) const {
    const uint4 w = __ldcg(reinterpret_cast<const uint4*>(row + i0));
    const uint32_t b[4] = {w.x, w.y, w.z, w.w};
    uint32_t k[4];
    bool any_nan = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t mag = b[e] & 0x7fffffffu;
      const bool isnan = mag > 0x7f800000u;
      const uint32_t x = mag ? b[e] : 0u;
      const uint32_t f = x ^ (static_cast<uint32_t>(static_cast<int32_t>(x) >> 31) | 0x80000000u);
      k[e] = isnan ? 0u : f;
      any_nan |= isnan;
    }
    nan |= any_nan;
    return make_uint4(k[0], k[1], k[2], k[3]);
  }
  // Keys of slots i0 .. i0+3 (i0 a multiple of 4 from lo, i0 < end).
  __device__ __forceinline__ uint4 fetch(int i0, int P, int end, bool& nan) const {
    float x[4];
    if (vec && i0 + 3 < end) {
      const float4 f = __ldcg(reinterpret_cast<const float4*>(row + i0));
      x[0] = f.x;
      x[1] = f.y;
      x[2] = f.z;
      x[3] = f.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = (i0 + e < end) ? __ldcg(row + i0 + e) : 0.f;
    }
    uint32_t k[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) k[e] = in_range(i0 + e, P, end) ? score_key(x[e], nan) : 0u;
    return make_uint4(k[0], k[1], k[2], k[3]);
  }
  // One bulk prefetch into L2 of the candidates' scores (the whole 16-byte
  // units inside [lo, end) of the row), so that the sample and the pass
  // mostly hit L2 instead of waiting on DRAM one round trip at a time.
  __device__ void prefetch(const Ctx& c) const {
    const uintptr_t a = (reinterpret_cast<uintptr_t>(row + c.lo) + 15) & ~static_cast<uintptr_t>(15);
    const uintptr_t b = reinterpret_cast<uintptr_t>(row + c.end) & ~static_cast<uintptr_t>(15);
    if (b > a) {
      uint64_t ga;
      asm volatile("cvta.to.global.u64 %0, %1;" : "=l"(ga) : "l"(static_cast<uint64_t>(a)));
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ga), "r"(static_cast<uint32_t>(b - a))
                   : "memory");
    }
  }
  __device__ void window(SSmem& sm, const Ctx& c, int need, int m, uint32_t& t_lo, uint32_t& t_hi) const {
    const float* r = row;
    sampled_window<1>(sm, c, need, m, [r](int slot) {
      bool ignored = false;  // NaN is flagged by the full pass
      return RunKeys<1>{{score_key(__ldcg(r + slot), ignored)}};
    }, t_lo, t_hi);
  }
};

// Philox-4x32-10 draws (Salmon et al., SC'11).
struct DrawKeys {
  static constexpr int U = 1;
  static constexpr bool GROUPED = false;
  static constexpr bool INTERIOR = false;
  static constexpr bool PREFETCH = false;
  uint4 ctr;  // counter words 1..3 (head + 65536 layer, seq, round)
  uint2 key;

  __device__ static DrawKeys make(const SelectParams& p, const Ctx&, int seq, int layer, int head) {
    DrawKeys k;
    // a shared draw (Random Attention, Appendix D's control) is the draw of
    // head 0 (of layer 0 for a whole sequence) used by every head
    if (p.draw_scope >= 1) head = 0;
    if (p.draw_scope >= 2) layer = 0;
    k.ctr = make_uint4(0u, static_cast<uint32_t>(head + 65536 * layer), static_cast<uint32_t>(seq), p.round);
    k.key = make_uint2(static_cast<uint32_t>(p.seed), static_cast<uint32_t>(p.seed >> 32));
    return k;
  }
  __device__ __forceinline__ uint4 fetch(int i0, int, int, bool&) const {
    return philox4x32_10(make_uint4(static_cast<uint32_t>(i0) >> 2, ctr.y, ctr.z, ctr.w), key);
  }
  __device__ void window(SSmem& sm, const Ctx&, int need, int m, uint32_t& t_lo, uint32_t& t_hi) const {
    if (threadIdx.x == 0) {
      // the need-th largest of m uniform draws, as a fraction of 2^32
      const double k = need, mm = m;
      const double mu = 1.0 - k / (mm + 1.0);
      const double sd = sqrt(k * (mm + 1.0 - k) / ((mm + 1.0) * (mm + 1.0) * (mm + 2.0)));
      const double wlo = mu - DRAW_SD * sd - 2.0 / (mm + 1.0), whi = mu + DRAW_SD * sd + 2.0 / (mm + 1.0);
      sm.t_lo = (wlo <= 0.0) ? 0u : static_cast<uint32_t>(wlo * 4294967296.0);
      sm.t_hi = (whi >= 1.0) ? 0xffffffffu : static_cast<uint32_t>(whi * 4294967296.0);
    }
    __syncthreads();
    t_lo = sm.t_lo;
    t_hi = sm.t_hi;
  }
};

// Final GQA scores, TriAttention paper summary, "Handling Grouped-Query
// Attention": the key of candidate i is the order-preserving u32 of
// max_g (S~(g)(i) - mean_g) / std_g over the group's G query heads, formed on
// the fly from the per-head scores [S][G][n_cap] and statistics [S][G][2].
template <int G>
struct ZMaxKeys {
  static constexpr int U = 1;
  static constexpr bool GROUPED = false;
  static constexpr bool INTERIOR = true;
  static constexpr bool PREFETCH = false;
  const float* base;  // row 0 of the G score rows
  int64_t n_cap;
  float mu[G], inv[G];
  bool vec;

  // score rows [block * G, block * G + G) and their statistics
  __device__ static ZMaxKeys at(const SelectParams& p, int64_t block) {
    ZMaxKeys k;
    k.n_cap = p.n_cap;
    k.base = p.scores + block * G * k.n_cap;
    k.vec = (reinterpret_cast<uintptr_t>(k.base) & 15) == 0 && (p.n_cap & 3) == 0;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      k.mu[g] = p.stats[(block * G + g) * 2];
      k.inv[g] = head_inv_std(p.stats[(block * G + g) * 2 + 1]);
    }
    return k;
  }
  __device__ static ZMaxKeys make(const SelectParams& p, const Ctx& c, int, int, int) { return at(p, c.s); }
  __device__ __forceinline__ float final_score(int slot) const {
    float best = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float z = head_z(__ldcg(base + g * n_cap + slot), mu[g], inv[g]);
      best = (g == 0) ? z : fmaxf(best, z);
    }
    return best;
  }
  // max_g z_g of slots i0 .. i0+3 (those < end; i0 a multiple of 4)
  __device__ __forceinline__ void best4(int i0, int end, float (&best)[4]) const {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float* row = base + g * n_cap;
      float x[4];
      if (vec && i0 + 3 < end) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(row + i0));
        x[0] = f.x;
        x[1] = f.y;
        x[2] = f.z;
        x[3] = f.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = (i0 + e < end) ? __ldcg(row + i0 + e) : 0.f;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float z = head_z(x[e], mu[g], inv[g]);
        best[e] = (g == 0) ? z : fmaxf(best[e], z);
      }
    }
  }
  // Keys of four slots that all lie in [P, end) (see ScoreKeys): the G
  // 16-byte loads first, then the same z-score maximum as best4 and
  // score_key's order in integer operations.
  // best4 for four slots inside the row (i0 + 3 < n_cap, vec): all G loads first
  __device__ __forceinline__ void best4_interior(int i0, float (&best)[4]) const {
    float4 f[G];
#pragma unroll
    for (int g = 0; g < G; ++g) f[g] = __ldcg(reinterpret_cast<const float4*>(base + g * n_cap + i0));
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float x[4] = {f[g].x, f[g].y, f[g].z, f[g].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float z = head_z(x[e], mu[g], inv[g]);
        best[e] = (g == 0) ? z : fmaxf(best[e], z);
      }
    }
  }
  __device__ __forceinline__ uint4 fetch_interior(int i0, bool& nan) const {
    float best[4];
    best4_interior(i0, best);
    uint32_t k[4];
    bool any_nan = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t b = __float_as_uint(best[e]);
      const uint32_t mag = b & 0x7fffffffu;
      const bool isnan = mag > 0x7f800000u;
      const uint32_t x = mag ? b : 0u;
      const uint32_t o = x ^ (static_cast<uint32_t>(static_cast<int32_t>(x) >> 31) | 0x80000000u);
      k[e] = isnan ? 0u : o;
      any_nan |= isnan;
    }
    nan |= any_nan;
    return make_uint4(k[0], k[1], k[2], k[3]);
  }
  __device__ __forceinline__ uint4 fetch(int i0, int P, int end, bool& nan) const {
    float best[4];
    best4(i0, end, best);
    uint32_t k[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) k[e] = in_range(i0 + e, P, end) ? score_key(best[e], nan) : 0u;
    return make_uint4(k[0], k[1], k[2], k[3]);
  }
  // max_g z_g of the 8 slots s0 .. s0+7 (s0 a multiple of 8, s0 + 7 < n_cap):
  // two 16-byte loads per head row when the rows are 16-byte aligned, so the
  // sample's loads do not crowd the load/store queue
  __device__ __forceinline__ void best8(int s0, float (&best)[8]) const {
    if (vec) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float4* q = reinterpret_cast<const float4*>(base + g * n_cap + s0);
        const float4 a = __ldcg(q), b = __ldcg(q + 1);
        const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float z = head_z(x[e], mu[g], inv[g]);
          best[e] = (g == 0) ? z : fmaxf(best[e], z);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) best[e] = final_score(s0 + e);
    }
  }
  __device__ void window(SSmem& sm, const Ctx& c, int need, int m, uint32_t& t_lo, uint32_t& t_hi) const {
    const ZMaxKeys& self = *this;
    sampled_window<8>(sm, c, need, m, [&self](int s0) {
      float best[8];
      self.best8(s0, best);
      RunKeys<8> o;
      bool ignored = false;
#pragma unroll
      for (int e = 0; e < 8; ++e) o.k[e] = score_key(best[e], ignored);
      return o;
    }, t_lo, t_hi);
  }
};

// Union-based selection across the H KV heads of a (seq, layer) (the
// TriAttention blog, "eviction (union-based selection)"): one keep list for
// the group. Candidates in the union of the heads' own top picks rank first,
// each group by the combined score max_h z_h (ZMaxKeys over the group's H
// score rows). Encoded in one u32 key: when the union holds at least `need`
// candidates only members compete (members: the score's order key, at least
// 1; others 0); otherwise every member is kept (key all ones) and the others
// compete by the combined score.
template <int H>
struct UnionKeys {
  static constexpr int U = 1;
  static constexpr bool GROUPED = true;
  static constexpr bool INTERIOR = true;
  static constexpr bool PREFETCH = false;
  ZMaxKeys<H> z;
  const uint32_t* member;  // the group's union bitmap, bit i = slot i
  bool many;
  bool vec;  // 16-byte loads allowed (z.vec)

  __device__ static UnionKeys make(const SelectParams& p, const Ctx& c, int, int, int) {
    UnionKeys k;
    const int64_t group = c.s / H;
    k.z = ZMaxKeys<H>::at(p, group);
    k.member = p.member + group * p.member_words;
    k.many = p.ucount[group] >= c.B - c.P - c.W;
    k.vec = k.z.vec;
    return k;
  }
  __device__ __forceinline__ uint32_t key(bool in_union, float comb, bool& nan) const {
    const uint32_t k = score_key(comb, nan);
    if (many) return in_union ? max(k, 1u) : 0u;
    return in_union ? 0xffffffffu : k;
  }
  // keys of four slots that all lie in [P, end) (no range checks)
  __device__ __forceinline__ uint4 fetch_interior(int i0, bool& nan) const {
    float best[4];
    z.best4_interior(i0, best);
    const uint32_t word = __ldg(member + (i0 >> 5)) >> (i0 & 31);  // i0 % 4 == 0: one word
    return make_uint4(key(word & 1u, best[0], nan), key((word >> 1) & 1u, best[1], nan),
                      key((word >> 2) & 1u, best[2], nan), key((word >> 3) & 1u, best[3], nan));
  }
  __device__ __forceinline__ uint4 fetch(int i0, int P, int end, bool& nan) const {
    float best[4];
    z.best4(i0, end, best);
    const uint32_t word = __ldg(member + (i0 >> 5)) >> (i0 & 31);  // i0 % 4 == 0: one word
    uint32_t k[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) k[e] = in_range(i0 + e, P, end) ? key((word >> e) & 1u, best[e], nan) : 0u;
    return make_uint4(k[0], k[1], k[2], k[3]);
  }
  __device__ void window(SSmem& sm, const Ctx& c, int need, int m, uint32_t& t_lo, uint32_t& t_hi) const {
    const UnionKeys& self = *this;
    sampled_window<8>(sm, c, need, m, [&self](int s0) {
      float best[8];
      self.z.best8(s0, best);
      const uint32_t word = __ldg(self.member + (s0 >> 5)) >> (s0 & 31);  // s0 % 8 == 0: one word
      RunKeys<8> o;
      bool ignored = false;
#pragma unroll
      for (int e = 0; e < 8; ++e) o.k[e] = self.key((word >> e) & 1u, best[e], ignored);
      return o;
    }, t_lo, t_hi);
  }
};

// One radix step over the short list or over all candidates (keys re-read
// or regenerated): histogram the digit of the keys still in play, pick the
// bin holding the need-th largest, narrow the state. Returns the bin count.
template <class Src>
__device__ unsigned radix_step(SSmem& sm, const Src& src, const Ctx& c, bool from_list, int nl, Radix& R,
                               bool& nan) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  sm.hist[0][t] = 0u;
  __syncthreads();
  if (from_list) {
    for (int e = t; e < nl; e += NT) {
      const uint32_t k = sm.lkey[e];
      if (R.matches(k)) atomicAdd(&sm.hist[0][R.digit(k)], 1u);
    }
  } else {
    for (int i0 = c.lo + 4 * t; i0 < c.end; i0 += 4 * NT) {
      const uint4 r = src.fetch(i0, c.P, c.end, nan);
      const uint32_t u[4] = {r.x, r.y, r.z, r.w};
      const uint32_t valid = valid_bits(i0, c.P, c.end);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (((valid >> e) & 1u) && R.matches(u[e])) atomicAdd(&sm.hist[0][R.digit(u[e])], 1u);
    }
  }
  __syncthreads();
  if (w == 0) pick_bin(sm, sm.hist[0], R.need, lane, 0);
  __syncthreads();
  const unsigned cnt = R.take(sm, 0);
  __syncthreads();  // pick fields and the histogram are rewritten next
  return cnt;
}

// Exact radix select: after it, the survivors are the keys with
// (k & mask) > prefix plus the first `need` (in slot order) with
// (k & mask) == prefix.
template <class Src>
__device__ void radix_select(SSmem& sm, const Src& src, const Ctx& c, bool from_list, int nl, uint32_t kmin,
                             uint32_t kmax, Radix& R, bool& nan) {
  R.start(kmin, kmax, R.need);
  while (!R.done) {
    const unsigned cnt = radix_step(sm, src, c, from_list, nl, R, nan);
    if (cnt == R.need || R.shift == 0) R.done = true; else R.next_digit();
  }
}

// The keep list of slice s (row s of p.keep), by the whole CTA. Every branch
// that returns early is uniform over the CTA.
template <class Src>
__device__ __forceinline__ void select_slice(const SelectParams& p, SSmem& sm, int64_t s) {
  const int t = threadIdx.x, lane = t & 31;
  Ctx c;
  c.s = s;
  c.n = p.n_valid[c.s];
  c.P = p.n_prompt;
  c.W = p.n_recent;
  c.B = p.budget;
  const int head = static_cast<int>(c.s % p.n_kv_heads);
  const int layer = static_cast<int>((c.s / p.n_kv_heads) % p.n_layers);
  const int seq = static_cast<int>(c.s / (static_cast<int64_t>(p.n_layers) * p.n_kv_heads));
  int32_t* keep = p.keep + c.s * static_cast<int64_t>(p.budget);

  if (c.n > p.n_cap || c.n < 0) {
    if (t == 0) set_status(p.dev_status, TRI_DEV_NVALID_OVER_CAP);
    return;
  }
  if (c.n <= c.B) {  // nothing to evict
    for (int j = t; j < c.B; j += NT) keep[j] = (j < c.n) ? j : -1;
    return;
  }
  c.end = c.n - c.W;
  c.lo = c.P & ~3;
  const int need_total = c.B - c.P - c.W;
  for (int j = t; j < c.P; j += NT) keep[j] = j;
  for (int j = t; j < c.W; j += NT) keep[c.B - c.W + j] = c.n - c.W + j;
  if (need_total == 0) return;
  const int m = c.end - c.P;  // candidates
  const Src src = Src::make(p, c, seq, layer, head);
  if constexpr (Src::PREFETCH) {
    if (t == 0) src.prefetch(c);
  }
  // the bitmaps cover every candidate: the pass fills them directly
  const bool direct = (c.end - c.lo) <= BM_SLOTS;
  bool nan = false;

  if (t == 0) {
    sm.nlist = 0u;
    sm.cnt_hi = 0u;
    sm.nan_seen = 0;
  }
  for (int j = t; j < BM_WORDS; j += NT) {
    sm.gt[j] = 0u;
    sm.eq[j] = 0u;
  }
  // ---- 1. window -----------------------------------------------------------
  uint32_t t_lo = 0u, t_hi = 0xffffffffu;
  if (m > LCAP) src.window(sm, c, need_total, m, t_lo, t_hi);
  __syncthreads();

  // ---- 2. one pass: count and mark keys above the window, list those in it -
  {
    const uint32_t win = t_hi - t_lo;
    unsigned hi = 0u;
    const int ng = (c.end - c.lo + 3) >> 2;
    constexpr int U = Src::U;
    // groups whose four slots all lie in [P, end): the first one from lo is
    // a partial group when P is not a multiple of 4, the last one when end
    // is not
    const int gin0 = (c.P > c.lo) ? 1 : 0, gin1 = ((c.end - c.lo) >> 2) - 1;
    for (int g0 = t; g0 < ng; g0 += NT * U) {
      uint4 r[U];
      uint32_t vm[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int g = g0 + j * NT;
        if (g < ng) {
          const int i0 = c.lo + 4 * g;
          bool inner = false;
          if constexpr (Src::INTERIOR) {
            inner = src.vec && g >= gin0 && g <= gin1;
            if (inner) r[j] = src.fetch_interior(i0, nan);
          }
          if (inner) {
            vm[j] = 0xfu;
          } else {
            r[j] = src.fetch(i0, c.P, c.end, nan);
            vm[j] = valid_bits(i0, c.P, c.end);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int g = g0 + j * NT;
        if (g >= ng) break;
        const int i0 = c.lo + 4 * g;
        const uint32_t u[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
        const uint32_t valid = vm[j];
        uint32_t nib = 0u, mid = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          nib |= static_cast<uint32_t>(u[e] > t_hi) << e;
          mid |= static_cast<uint32_t>(u[e] - t_lo <= win) << e;
        }
        nib &= valid;
        mid &= valid & ~nib;
        if (mid) {  // a key inside the window joins the short list
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if ((mid >> e) & 1u) {
              const unsigned at = atomicAdd(&sm.nlist, 1u);
              if (at < LCAP) {
                sm.lkey[at] = u[e];
                sm.lslot[at] = i0 + e;
              }
            }
          }
        }
        if (nib) {
          hi += __popc(nib);
          const int rel = i0 - c.lo;  // multiple of 4: the nibble stays inside one word
          if (direct) atomicOr(&sm.gt[rel >> 5], nib << (rel & 31));
        }
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) hi += __shfl_xor_sync(FULL_MASK, hi, o);
    if (lane == 0 && hi) atomicAdd(&sm.cnt_hi, hi);
  }
  __syncthreads();

  // ---- 3. the exact threshold ------------------------------------------------
  const unsigned chi = sm.cnt_hi, nl = sm.nlist;
  const unsigned need0 = static_cast<unsigned>(need_total);
  const bool fast = (nl <= LCAP) && (chi < need0) && (need0 <= chi + nl);
  Radix R;
  if (fast) {
    // the threshold is among the listed keys
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int e = t; e < static_cast<int>(nl); e += NT) {
      kmin = min(kmin, sm.lkey[e]);
      kmax = max(kmax, sm.lkey[e]);
    }
    block_minmax(sm, kmin, kmax);
    R.need = need0 - chi;
    radix_select(sm, src, c, true, static_cast<int>(nl), kmin, kmax, R, nan);
    if (direct) {
      for (int e = t; e < static_cast<int>(nl); e += NT) {
        const uint32_t k = sm.lkey[e] & R.mask;
        const int rel = sm.lslot[e] - c.lo;
        if (k > R.prefix) atomicOr(&sm.gt[rel >> 5], 1u << (rel & 31));
        if (k == R.prefix) atomicOr(&sm.eq[rel >> 5], 1u << (rel & 31));
      }
    }
  } else {
    // the window missed: exact radix select over every candidate
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int i0 = c.lo + 4 * t; i0 < c.end; i0 += 4 * NT) {
      const uint4 r = src.fetch(i0, c.P, c.end, nan);
      const uint32_t u[4] = {r.x, r.y, r.z, r.w};
      const uint32_t valid = valid_bits(i0, c.P, c.end);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if ((valid >> e) & 1u) {
          kmin = min(kmin, u[e]);
          kmax = max(kmax, u[e]);
        }
      }
    }
    block_minmax(sm, kmin, kmax);
    R.need = need0;
    radix_select(sm, src, c, false, 0, kmin, kmax, R, nan);
    t_lo = 0u;  // every key is "in the window" for the emission below
    t_hi = 0xffffffffu;
  }
  __syncthreads();

  // ---- 4. emission, one bitmap-sized piece at a time --------------------------
  // keep = keys above t_hi, plus keys in [t_lo, t_hi] with (k & mask) >
  // prefix, plus the first `need` in slot order of the keys in [t_lo, t_hi]
  // with (k & mask) == prefix. (The radix state only ranks keys inside the
  // window; a key outside it may share the prefix bits.)
  const bool built = fast && direct;
  const uint32_t win = t_hi - t_lo;
  unsigned eq_left = R.need, out = 0u;
  for (int base = c.lo; base < c.end; base += BM_SLOTS) {
    const int pend = min(c.end, base + BM_SLOTS);
    const int words = (pend - base + 31) / 32;
    if (!built) {
      for (int j = t; j < words; j += NT) {
        sm.gt[j] = 0u;
        sm.eq[j] = 0u;
      }
      __syncthreads();
      for (int i0 = base + 4 * t; i0 < pend; i0 += 4 * NT) {
        const uint4 r = src.fetch(i0, c.P, c.end, nan);
        const uint32_t u[4] = {r.x, r.y, r.z, r.w};
        const uint32_t valid = valid_bits(i0, c.P, pend);
        uint32_t ng = 0u, ne = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t k = u[e] & R.mask;
          const bool in_win = u[e] - t_lo <= win;
          ng |= static_cast<uint32_t>(u[e] > t_hi || (in_win && k > R.prefix)) << e;
          ne |= static_cast<uint32_t>(in_win && k == R.prefix) << e;
        }
        ng &= valid;
        ne &= valid;
        const int rel = i0 - base;
        if (ng) atomicOr(&sm.gt[rel >> 5], ng << (rel & 31));
        if (ne) atomicOr(&sm.eq[rel >> 5], ne << (rel & 31));
      }
      __syncthreads();
    }
    // rank the equal slots in slot order; keep the first eq_left of them
    const int wpt = (words + NT - 1) / NT;  // words per thread, contiguous
    const int w0 = min(words, t * wpt), w1 = min(words, w0 + wpt);
    unsigned ce = 0u;
    for (int j = w0; j < w1; ++j) ce += __popc(sm.eq[j]);
    unsigned tot_eq;
    unsigned r_eq = block_scan(sm, ce, &tot_eq);
    unsigned ck = 0u;
    for (int j = w0; j < w1; ++j) {
      uint32_t e = sm.eq[j], kept = 0u;
      while (e) {
        const int b = __ffs(e) - 1;
        e &= e - 1u;
        if (r_eq < eq_left) kept |= 1u << b;
        ++r_eq;
      }
      sm.eq[j] = kept | sm.gt[j];  // final keep mask of the word
      ck += __popc(sm.eq[j]);
    }
    eq_left = (tot_eq >= eq_left) ? 0u : eq_left - tot_eq;
    unsigned tot_keep;
    unsigned r = out + block_scan(sm, ck, &tot_keep);
    for (int j = w0; j < w1; ++j) {
      uint32_t k = sm.eq[j];
      while (k) {
        const int b = __ffs(k) - 1;
        k &= k - 1u;
        if (r < need0) keep[c.P + r] = base + 32 * j + b;
        ++r;
      }
    }
    out += tot_keep;
    __syncthreads();
  }
  if (nan) atomicOr(&sm.nan_seen, 1);
  __syncthreads();
  if (t == 0 && sm.nan_seen) set_status(p.dev_status, TRI_DEV_NAN_SCORE);
}

// One CTA per slice, or per group of p.group consecutive slices for a key
// source whose keep list is shared (Src::GROUPED): the group's first slice is
// selected and its list copied to the others.
template <class Src>
__global__ void __launch_bounds__(NT, MINB) select_kernel(const __grid_constant__ SelectParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SSmem& sm = *reinterpret_cast<SSmem*>(smem_raw);
  const int64_t s = Src::GROUPED ? static_cast<int64_t>(blockIdx.x) * p.group : blockIdx.x;
  select_slice<Src>(p, sm, s);
  if (Src::GROUPED) {
    __syncthreads();
    const int32_t* k0 = p.keep + s * static_cast<int64_t>(p.budget);
    for (int h = 1; h < p.group; ++h) {
      int32_t* kh = p.keep + (s + h) * static_cast<int64_t>(p.budget);
      for (int j = threadIdx.x; j < p.budget; j += NT) kh[j] = k0[j];
    }
  }
}

}  // namespace
}  // namespace tri
