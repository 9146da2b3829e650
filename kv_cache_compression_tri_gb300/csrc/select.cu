// select.cu -- per-slice budgeted top-k selection in one CTA.
//
// TriAttention paper summary, "Retention and eviction" (top-B by score);
// Random Attention, Eq. 2 (top-K with the prompt forced in): keep [0, P) U
// top-(B-P-W) candidates U [n-W, n), ascending. One CTA of 1024 threads owns
// one slice:
//   1. candidate keys -- the order-preserving u32 of the fp32 score -- are
//      staged in shared memory (up to 32768,
//      128 KB), slot-ordered; warp w owns slots [1024 w, 1024 w + 1024) and
//      lane l reads slot 1024 w + 32 q + l at step q (conflict-free);
//   2. the block finds the keys' min and max: bits above the highest bit
//      where they differ are common to all keys, so the first 8-bit radix
//      digit starts just below them and spans the keys' real range; one
//      histogram pass (per-warp private histograms, plain shared atomics)
//      finds the digit bin holding the k-th largest key;
//   3. the keys of that bin (a few hundred typically) are collected into a
//      short list and the remaining digits are resolved on the list only;
//      the select stops as soon as a bin is taken whole;
//   4. emission in slot order: each lane keeps one bit per step for "above
//      the threshold" and "equal to it"; warp ballots give ranks inside a
//      warp and a 32-entry scan of warp totals gives the warp's offset, so
//      the keep list comes out ascending without sorting; among keys equal
//      to the threshold the lower slots win.
// Slices with more than 32768 candidates, or whose threshold bin does not
// fit the list, fall back to full-array radix passes (re-staging the keys
// for every pass when they do not fit shared memory). The Random Attention
// draws have their own kernel (rand_select.cu).
#include <cuda_runtime.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

// Launch geometry: NT threads, up to KCAP keys staged per super-chunk; warp w
// owns slots [WSPAN w, WSPAN (w+1)) of a super-chunk and lane l reads slot
// WSPAN w + 32 q + l at step q.
template <int NT_, int KCAP_, int LCAP_, int MINB_>
struct SelGeo {
  static constexpr int NT = NT_;
  static constexpr int MINB = MINB_;  // CTAs per SM the registers must allow
  static constexpr int NW = NT / 32;
  static constexpr int KCAP = KCAP_;
  static constexpr int WSPAN = KCAP / NW;
  static constexpr int NQ = WSPAN / 32;
  static constexpr int LCAP = LCAP_;  // short-list capacity
  static constexpr size_t SMEM = KCAP * sizeof(uint32_t)          // keys
                                 + NW * 256 * sizeof(unsigned)     // per-warp histograms
                                 + LCAP * sizeof(uint32_t);        // short list
  static_assert(NQ == 32 && WSPAN % 128 == 0, "select geometry");
};
using BigGeo = SelGeo<1024, 32768, 4096, 1>;  // 32K-row slices: one CTA per SM
using SmallGeo = SelGeo<256, 8192, 1024, 4>;  // short slices: four CTAs per SM

struct SliceCtx {
  int64_t s;
  int n, P, W, B;
  int lo;   // first slot of the staged range (P rounded down to 4)
  int end;  // n - W: exclusive end of the candidates
  int seq, layer, head;
};

template <int NW>
struct Smem {
  unsigned hist[256];
  unsigned wtot[NW];
  unsigned wmin[NW], wmax[NW];
  int pick_digit;
  unsigned pick_above, pick_count;
  unsigned nlist;
  int nan_seen;
};

__device__ __forceinline__ bool in_range(int i, int lo, int hi) {
  return static_cast<unsigned>(i - lo) < static_cast<unsigned>(hi - lo);
}

// Stage the keys of slots [base, base + KCAP) into skey (slot-ordered).
// Slots outside [P, end) get key 0 and are masked out by their index later.
// Accumulates this thread's min / max over the valid keys it staged.
template <class G>
__device__ __forceinline__ void stage_keys(const SelectParams& p, const SliceCtx& c, int base,
                                           uint32_t* skey, bool& nan, uint32_t& kmin, uint32_t& kmax) {
  constexpr int WSPAN = G::WSPAN;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int V = WSPAN / 4 / 32;  // 16-byte groups per lane (8)
  const float* row = p.scores + c.s * static_cast<int64_t>(p.n_cap);
  const bool vec = ((c.s * static_cast<int64_t>(p.n_cap) + base) & 3) == 0;
  float4 f[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int g = w * (WSPAN / 4) + v * 32 + lane;
    const int i0 = base + 4 * g;
    if (vec && i0 + 3 < c.end) {
      f[v] = __ldcg(reinterpret_cast<const float4*>(row + i0));
    } else {
      f[v] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i0 < c.end) f[v].x = __ldcg(row + i0);
      if (i0 + 1 < c.end) f[v].y = __ldcg(row + i0 + 1);
      if (i0 + 2 < c.end) f[v].z = __ldcg(row + i0 + 2);
      if (i0 + 3 < c.end) f[v].w = __ldcg(row + i0 + 3);
    }
  }
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int g = w * (WSPAN / 4) + v * 32 + lane;
    const int i0 = base + 4 * g;
    const float x[4] = {f[v].x, f[v].y, f[v].z, f[v].w};
    uint32_t k[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool valid = in_range(i0 + e, c.P, c.end);
      k[e] = valid ? score_key(x[e], nan) : 0u;
      if (valid) {
        kmin = min(kmin, k[e]);
        kmax = max(kmax, k[e]);
      }
    }
    reinterpret_cast<uint4*>(skey)[g] = make_uint4(k[0], k[1], k[2], k[3]);
  }
}

// Warp 0 finds digit b with count(digits > b) < need <= count(digits >= b)
// and publishes (b, count above b, count of b). Caller syncs around it.
template <class SM>
__device__ __forceinline__ void pick_bin(SM& sm, unsigned need, int lane) {
  unsigned h[8], ls = 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = sm.hist[lane * 8 + j];
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
        sm.pick_digit = lane * 8 + j;
        sm.pick_above = cum;
        sm.pick_count = h[j];
        break;
      }
      cum += h[j];
    }
  }
}

// Exclusive prefix of this warp's entry among the 32 warp totals in
// sm.wtot, and the grand total (every warp computes it redundantly).
template <int NW>
__device__ __forceinline__ unsigned warp_offset(const Smem<NW>& sm, int w, int lane, unsigned& total) {
  const unsigned x = (lane < NW) ? sm.wtot[lane] : 0u;
  unsigned incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += y;
  }
  total = __shfl_sync(FULL_MASK, incl, 31);
  return __shfl_sync(FULL_MASK, incl - x, w);
}

template <class G>
__global__ void __launch_bounds__(G::NT, G::MINB) select_kernel(const __grid_constant__ SelectParams p) {
  constexpr int NT = G::NT, NW = G::NW, KCAP = G::KCAP, WSPAN = G::WSPAN, NQ = G::NQ, LCAP = G::LCAP;
  extern __shared__ __align__(16) uint32_t skey[];
  unsigned* whist = skey + KCAP;  // [NW][256]
  uint32_t* lkey = whist + NW * 256;
  __shared__ Smem<NW> sm;

  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  SliceCtx c;
  c.s = blockIdx.x;
  c.n = p.n_valid[c.s];
  c.P = p.n_prompt;
  c.W = p.n_recent;
  c.B = p.budget;
  const int lhc = p.n_layers * p.n_kv_heads;
  c.head = static_cast<int>(c.s % p.n_kv_heads);
  c.layer = static_cast<int>((c.s / p.n_kv_heads) % p.n_layers);
  c.seq = static_cast<int>(c.s / lhc);
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

  const int n_super = (c.end - c.lo + KCAP - 1) / KCAP;
  const bool staged_once = (n_super == 1);
  if (t == 0) {
    sm.nan_seen = 0;
    sm.nlist = 0u;
  }
  bool nan = false;
  uint32_t prefix = 0u, mask = 0u;
  int shift = 24;  // lowest bit of the next digit
  int width = 8;   // bits of the next digit
  unsigned need = static_cast<unsigned>(need_total);
  bool exact = false, resolved = false;
  const int wbase_slot = w * WSPAN + lane;  // slot offset of (warp, lane) at step 0

  if (staged_once) {
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    stage_keys<G>(p, c, c.lo, skey, nan, kmin, kmax);
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
    const uint32_t diff = kmin ^ kmax;
    if (diff == 0u) {
      prefix = kmin;  // all candidates equal: lowest slots win
      mask = 0xffffffffu;
      resolved = true;
    } else {
      const int hb = 31 - __clz(diff);
      shift = max(hb - 7, 0);
      width = hb - shift + 1;
      mask = (hb == 31) ? 0u : ~((2u << hb) - 1u);  // bits above hb: common to all keys
      prefix = kmin & mask;
    }
  }

  // ---- radix passes over the full key array -------------------------------
  unsigned* my_hist = whist + w * 256;
  while (!resolved) {
    for (int b = lane; b < 256; b += 32) my_hist[b] = 0u;
    __syncwarp();
    const uint32_t dmask = (1u << width) - 1u;
    for (int sc = 0; sc < n_super; ++sc) {
      const int base = c.lo + sc * KCAP;
      if (!staged_once) {
        uint32_t a = 0xffffffffu, b = 0u;
        __syncthreads();  // previous users of skey are done
        stage_keys<G>(p, c, base, skey, nan, a, b);
        __syncthreads();
      }
#pragma unroll 8
      for (int q = 0; q < NQ; ++q) {
        const int j = wbase_slot + q * 32;
        const uint32_t k = skey[j];
        if (in_range(base + j, c.P, c.end) && (k & mask) == prefix) atomicAdd(&my_hist[(k >> shift) & dmask], 1u);
      }
    }
    __syncthreads();
    for (int b = t; b < 256; b += NT) {
      unsigned sum = 0u;
#pragma unroll 8
      for (int ww = 0; ww < NW; ++ww) sum += whist[ww * 256 + b];
      sm.hist[b] = sum;
    }
    __syncthreads();
    if (w == 0) pick_bin(sm, need, lane);
    __syncthreads();
    const unsigned bsel = static_cast<unsigned>(sm.pick_digit);
    need -= sm.pick_above;
    const unsigned cnt = sm.pick_count;
    prefix |= bsel << shift;
    mask |= dmask << shift;
    __syncthreads();  // pick_* and the histograms are rewritten next
    if (cnt == need) {
      exact = true;  // every key with this prefix is kept
      resolved = true;
    } else if (shift == 0) {
      resolved = true;  // full key known; ties at it are ranked by slot
    } else {
      width = min(8, shift);
      shift -= width;
      if (staged_once && cnt <= LCAP) break;  // finish on the short list
    }
  }

  // ---- finish on the short list of keys sharing the current prefix ---------
  if (!resolved) {
#pragma unroll 4
    for (int q = 0; q < NQ; ++q) {
      const int j = wbase_slot + q * 32;
      const uint32_t k = skey[j];
      const bool m = in_range(c.lo + j, c.P, c.end) && ((k & mask) == prefix);
      const unsigned bal = __ballot_sync(FULL_MASK, m);
      if (bal) {
        unsigned at = 0u;
        if (lane == 0) at = atomicAdd(&sm.nlist, static_cast<unsigned>(__popc(bal)));
        at = __shfl_sync(FULL_MASK, at, 0);
        if (m) {
          at += __popc(bal & ((1u << lane) - 1u));
          lkey[at] = k;
        }
      }
    }
    __syncthreads();
    const int nl = static_cast<int>(sm.nlist);
    while (!resolved) {
      for (int b = t; b < 256; b += NT) sm.hist[b] = 0u;
      __syncthreads();
      const uint32_t dmask = (1u << width) - 1u;
      for (int e = t; e < nl; e += NT) {
        const uint32_t k = lkey[e];
        if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & dmask], 1u);
      }
      __syncthreads();
      if (w == 0) pick_bin(sm, need, lane);
      __syncthreads();
      const unsigned bsel = static_cast<unsigned>(sm.pick_digit);
      need -= sm.pick_above;
      const unsigned cnt = sm.pick_count;
      prefix |= bsel << shift;
      mask |= dmask << shift;
      __syncthreads();
      if (cnt == need) {
        exact = true;
        resolved = true;
      } else if (shift == 0) {
        resolved = true;
      } else {
        width = min(8, shift);
        shift -= width;
      }
    }
  }

  // ---- emission in slot order --------------------------------------------
  // keep(i) = (k & mask) > prefix, or == prefix and (exact, or its rank among
  // the threshold-equal keys in slot order is < need).
  const unsigned lt_mask = (1u << lane) - 1u;
  unsigned eq_carry = 0u, keep_carry = 0u;
  for (int sc = 0; sc < n_super; ++sc) {
    const int base = c.lo + sc * KCAP;
    if (!staged_once) {
      uint32_t a = 0xffffffffu, b = 0u;
      __syncthreads();
      stage_keys<G>(p, c, base, skey, nan, a, b);
      __syncthreads();
    }
    uint32_t eqb = 0u, gtb = 0u;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int j = wbase_slot + q * 32;
      const uint32_t k = skey[j] & mask;
      const bool valid = in_range(base + j, c.P, c.end);
      gtb |= static_cast<uint32_t>(valid && k > prefix) << q;
      eqb |= static_cast<uint32_t>(valid && k == prefix) << q;
    }
    if (!exact) {
      unsigned cnt = 0u;
#pragma unroll
      for (int q = 0; q < NQ; ++q) cnt += __popc(__ballot_sync(FULL_MASK, (eqb >> q) & 1u));
      if (lane == 0) sm.wtot[w] = cnt;
      __syncthreads();
      unsigned total_eq;
      unsigned rank = eq_carry + warp_offset(sm, w, lane, total_eq);
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const unsigned bq = __ballot_sync(FULL_MASK, (eqb >> q) & 1u);
        if (((eqb >> q) & 1u) && rank + __popc(bq & lt_mask) >= need) eqb &= ~(1u << q);
        rank += __popc(bq);
      }
      eq_carry += total_eq;
      __syncthreads();  // sm.wtot is rewritten below
    }
    const uint32_t kb = gtb | eqb;
    unsigned cnt = 0u;
#pragma unroll
    for (int q = 0; q < NQ; ++q) cnt += __popc(__ballot_sync(FULL_MASK, (kb >> q) & 1u));
    if (lane == 0) sm.wtot[w] = cnt;
    __syncthreads();
    unsigned total_keep;
    unsigned rank = keep_carry + warp_offset(sm, w, lane, total_keep);
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const unsigned bq = __ballot_sync(FULL_MASK, (kb >> q) & 1u);
      const unsigned r = rank + __popc(bq & lt_mask);
      if (((kb >> q) & 1u) && r < static_cast<unsigned>(need_total)) keep[c.P + r] = base + wbase_slot + q * 32;
      rank += __popc(bq);
    }
    keep_carry += total_keep;
    __syncthreads();
  }
  if (nan) atomicOr(&sm.nan_seen, 1);
  __syncthreads();
  if (t == 0 && sm.nan_seen) set_status(p.dev_status, TRI_DEV_NAN_SCORE);
}

template <class G>
cudaError_t launch_geo(const SelectParams& p, int n_slices, cudaStream_t st) {
  // The dynamic shared memory opt-in is a per-device function attribute;
  // setting it on every call is cheap and covers every device.
  const cudaError_t e = cudaFuncSetAttribute(select_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(G::SMEM));
  if (e != cudaSuccess) return e;
  select_kernel<G><<<n_slices, G::NT, G::SMEM, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select(const SelectParams& p, int n_slices, cudaStream_t st) {
  // The candidate span [P rounded down to 4, n_valid - W) of any slice is at
  // most n_cap - W - (P & ~3) slots; short slices take the small geometry.
  const int64_t span = static_cast<int64_t>(p.n_cap) - p.n_recent - (p.n_prompt & ~3);
  if (span <= SmallGeo::KCAP) return launch_geo<SmallGeo>(p, n_slices, st);
  return launch_geo<BigGeo>(p, n_slices, st);
}

}  // namespace tri
