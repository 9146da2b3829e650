// rand_select.cu -- Random Attention keep lists without a score.
//
// Random Attention, section 3 (Eq. 3, Algorithm 1): the prompt is kept, every
// other candidate draws an i.i.d. uniform u_i (word i mod 4 of
// Philox-4x32-10 with counter (i/4, head + 65536 layer, seq, round) and key =
// the seed), and the top (B - P - W) draws survive, ties to the lower slot;
// the recent buffer is kept unscored (section 2).
//
// Because the draws are i.i.d. uniform, the need-th largest of m of them is
// known in distribution: its position in [0, 1) has mean 1 - k/(m+1) and
// variance k (m+1-k) / ((m+1)^2 (m+2)) (an order statistic of uniforms). One
// CTA per slice:
//   1. one Philox sweep counts the draws above a window of +-8 standard
//      deviations around that mean (their slots go to a bitmap) and collects
//      the draws inside the window (about 16 sd x m of them, ~900 for the
//      32K-candidate workloads) into a short list;
//   2. if the threshold provably lies in the window (count above < need <=
//      count above + list size) the exact threshold and the number of draws
//      equal to it still needed are found by a radix select on the list only;
//      otherwise (never seen for uniform draws, but handled exactly) a radix
//      select over all draws, regenerated per pass, finds them;
//   3. emission from bitmaps of "above" and "equal" slots in slot order
//      (per-thread popcounts and one block scan), the equal ones ranked by
//      slot, so the keep list is ascending without sorting.
// Shared memory stays small (bitmaps for 65536 slots + the list), so six
// CTAs share an SM and their phases overlap. Slices with more candidates
// than the bitmaps cover are emitted in bitmap-sized pieces.
#include <cuda_runtime.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

constexpr int RT = 256;             // threads per CTA
constexpr int RW = RT / 32;         // warps
constexpr int BM_SLOTS = 65536;     // slots covered by one pair of bitmaps
constexpr int BM_WORDS = BM_SLOTS / 32;
constexpr int RLCAP = 2048;         // short-list capacity

struct RSmem {
  uint32_t gt[BM_WORDS];  // slot above the threshold
  uint32_t eq[BM_WORDS];  // slot equal to the threshold (candidate tie)
  uint32_t lkey[RLCAP];
  int32_t lslot[RLCAP];
  unsigned hist[256];
  unsigned wsum[RW];
  unsigned nlist;
  unsigned cnt_hi;
  uint32_t t_lo, t_hi;
  int pick_digit;
  unsigned pick_above, pick_count;
  unsigned total;
};

struct RCtx {
  int64_t s;
  int n, P, W, B, lo, end;
  uint4 ctr;  // counter words 1..3 (head + 65536 layer, seq, round)
  uint2 key;
};

__device__ __forceinline__ bool in_range(int i, int lo, int hi) {
  return static_cast<unsigned>(i - lo) < static_cast<unsigned>(hi - lo);
}

__device__ __forceinline__ uint4 draws(const RCtx& c, int i0) {
  return philox4x32_10(make_uint4(static_cast<uint32_t>(i0) >> 2, c.ctr.y, c.ctr.z, c.ctr.w), c.key);
}

// Block-wide exclusive scan of one value per thread; returns the thread's
// offset, and the total in *total.
__device__ __forceinline__ unsigned block_scan(RSmem& sm, unsigned v, unsigned* total) {
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
    const unsigned x = (lane < RW) ? sm.wsum[lane] : 0u;
    unsigned xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(FULL_MASK, xi, o);
      if (lane >= o) xi += y;
    }
    if (lane < RW) sm.wsum[lane] = xi - x;
    if (lane == 31) sm.total = xi;
  }
  __syncthreads();
  const unsigned off = incl - v + sm.wsum[w];
  *total = sm.total;
  __syncthreads();
  return off;
}

// digit b with count(digits > b) < need <= count(digits >= b), by warp 0
__device__ __forceinline__ void pick_bin(RSmem& sm, unsigned need, int lane) {
  unsigned h[8], ls = 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = sm.hist[lane * 8 + j];
    ls += h[j];
  }
  unsigned suf = ls;
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

// One radix step over either the short list (from_list) or all draws
// (regenerated): histogram the 8-bit digit at `shift` of keys matching
// (prefix, mask), pick the bin, narrow (prefix, mask, need). Returns the
// count of the picked bin.
__device__ unsigned radix_step(RSmem& sm, const RCtx& c, bool from_list, int nl, int shift,
                               uint32_t& prefix, uint32_t& mask, unsigned& need) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  if (t < 256) sm.hist[t] = 0u;
  __syncthreads();
  if (from_list) {
    for (int e = t; e < nl; e += RT) {
      const uint32_t k = sm.lkey[e];
      if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & 0xffu], 1u);
    }
  } else {
    for (int i0 = c.lo + 4 * t; i0 < c.end; i0 += 4 * RT) {
      const uint4 r = draws(c, i0);
      const uint32_t u[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (in_range(i0 + e, c.P, c.end) && (u[e] & mask) == prefix)
          atomicAdd(&sm.hist[(u[e] >> shift) & 0xffu], 1u);
    }
  }
  __syncthreads();
  if (w == 0) pick_bin(sm, need, lane);
  __syncthreads();
  need -= sm.pick_above;
  const unsigned cnt = sm.pick_count;
  prefix |= static_cast<uint32_t>(sm.pick_digit) << shift;
  mask |= 0xffu << shift;
  __syncthreads();
  return cnt;
}

__global__ void __launch_bounds__(RT, 6) rand_select_kernel(const __grid_constant__ SelectParams p) {
  extern __shared__ __align__(16) unsigned char rsmem_raw[];
  RSmem& sm = *reinterpret_cast<RSmem*>(rsmem_raw);
  const int t = threadIdx.x, lane = t & 31;
  RCtx c;
  c.s = blockIdx.x;
  c.n = p.n_valid[c.s];
  c.P = p.n_prompt;
  c.W = p.n_recent;
  c.B = p.budget;
  const int head = static_cast<int>(c.s % p.n_kv_heads);
  const int layer = static_cast<int>((c.s / p.n_kv_heads) % p.n_layers);
  const int seq = static_cast<int>(c.s / (static_cast<int64_t>(p.n_layers) * p.n_kv_heads));
  c.ctr = make_uint4(0u, static_cast<uint32_t>(head + 65536 * layer), static_cast<uint32_t>(seq), p.round);
  c.key = make_uint2(static_cast<uint32_t>(p.seed), static_cast<uint32_t>(p.seed >> 32));
  int32_t* keep = p.keep + c.s * static_cast<int64_t>(p.budget);

  if (c.n > p.n_cap || c.n < 0) {
    if (t == 0) set_status(p.dev_status, TRI_DEV_NVALID_OVER_CAP);
    return;
  }
  if (c.n <= c.B) {
    for (int j = t; j < c.B; j += RT) keep[j] = (j < c.n) ? j : -1;
    return;
  }
  c.end = c.n - c.W;
  c.lo = c.P & ~3;
  const int need_total = c.B - c.P - c.W;
  for (int j = t; j < c.P; j += RT) keep[j] = j;
  for (int j = t; j < c.W; j += RT) keep[c.B - c.W + j] = c.n - c.W + j;
  if (need_total == 0) return;
  const int m = c.end - c.P;
  const bool fits = (c.end - c.lo) <= BM_SLOTS;

  uint32_t prefix = 0u, mask = 0u;
  unsigned need = static_cast<unsigned>(need_total);
  bool fast = false;
  if (fits) {
    if (t == 0) {
      // window around the need-th largest of m uniform draws (as a fraction)
      const double k = need_total, mm = m;
      const double mu = 1.0 - k / (mm + 1.0);
      const double sd = sqrt(k * (mm + 1.0 - k) / ((mm + 1.0) * (mm + 1.0) * (mm + 2.0)));
      const double wlo = mu - 8.0 * sd - 2.0 / (mm + 1.0), whi = mu + 8.0 * sd + 2.0 / (mm + 1.0);
      sm.t_lo = (wlo <= 0.0) ? 0u : static_cast<uint32_t>(wlo * 4294967296.0);
      sm.t_hi = (whi >= 1.0) ? 0xffffffffu : static_cast<uint32_t>(whi * 4294967296.0);
      sm.nlist = 0u;
      sm.cnt_hi = 0u;
    }
    for (int j = t; j < BM_WORDS; j += RT) {
      sm.gt[j] = 0u;
      sm.eq[j] = 0u;
    }
    __syncthreads();
    const uint32_t t_lo = sm.t_lo, t_hi = sm.t_hi;
    unsigned hi = 0u;
    const uint32_t win = t_hi - t_lo;
    for (int i0 = c.lo + 4 * t; i0 < c.end; i0 += 4 * RT) {
      const uint4 r = draws(c, i0);
      const uint32_t u[4] = {r.x, r.y, r.z, r.w};
      uint32_t valid = 0xfu;  // only the first and last groups hold non-candidates
      if (i0 < c.P || i0 + 3 >= c.end) {
        valid = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) valid |= static_cast<uint32_t>(in_range(i0 + e, c.P, c.end)) << e;
      }
      uint32_t nib = 0u, mid = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        nib |= static_cast<uint32_t>(u[e] > t_hi) << e;
        mid |= static_cast<uint32_t>(u[e] - t_lo <= win) << e;
      }
      nib &= valid;
      mid &= valid & ~nib;
      if (mid) {  // rare: a draw inside the window joins the short list
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if ((mid >> e) & 1u) {
            const unsigned at = atomicAdd(&sm.nlist, 1u);
            if (at < RLCAP) {
              sm.lkey[at] = u[e];
              sm.lslot[at] = i0 + e;
            }
          }
        }
      }
      if (nib) {
        const int rel = i0 - c.lo;  // multiple of 4: the nibble stays inside one word
        atomicOr(&sm.gt[rel >> 5], nib << (rel & 31));
        hi += __popc(nib);
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) hi += __shfl_xor_sync(FULL_MASK, hi, o);
    if (lane == 0) atomicAdd(&sm.cnt_hi, hi);
    __syncthreads();
    const unsigned chi = sm.cnt_hi, nl = sm.nlist;
    fast = (nl <= RLCAP) && (chi < need) && (need <= chi + nl);
    if (fast) {
      need -= chi;  // the threshold is among the list's draws
      for (int shift = 24; shift >= 0; shift -= 8) {
        const unsigned cnt = radix_step(sm, c, true, static_cast<int>(nl), shift, prefix, mask, need);
        if (cnt == need) break;
      }
      // draws above the window are already in the "above" bitmap; add the
      // list's draws above the threshold and mark the ones equal to it
      for (int e = t; e < static_cast<int>(nl); e += RT) {
        const uint32_t k = sm.lkey[e] & mask;
        const int rel = sm.lslot[e] - c.lo;
        if (k > prefix) atomicOr(&sm.gt[rel >> 5], 1u << (rel & 31));
        if (k == prefix) atomicOr(&sm.eq[rel >> 5], 1u << (rel & 31));
      }
      __syncthreads();
    }
  }
  if (!fast) {
    prefix = 0u;
    mask = 0u;
    need = static_cast<unsigned>(need_total);
    for (int shift = 24; shift >= 0; shift -= 8) {
      const unsigned cnt = radix_step(sm, c, false, 0, shift, prefix, mask, need);
      if (cnt == need) break;
    }
  }
  // Here: keep = draws with (u & mask) > prefix, plus the first `need` (in
  // slot order) with (u & mask) == prefix.

  // ---- emission, one bitmap-sized piece at a time --------------------------
  // (the fast path has its single piece's bitmaps built already; otherwise
  // each piece's bitmaps are rebuilt from regenerated draws)
  unsigned eq_left = need, out = 0u;
  for (int base = c.lo; base < c.end; base += BM_SLOTS) {
    const int pend = min(c.end, base + BM_SLOTS);
    const int words = (pend - base + 31) / 32;
    if (!fast) {
      for (int j = t; j < words; j += RT) {
        sm.gt[j] = 0u;
        sm.eq[j] = 0u;
      }
      __syncthreads();
      for (int i0 = base + 4 * t; i0 < pend; i0 += 4 * RT) {
        const uint4 r = draws(c, i0);
        const uint32_t u[4] = {r.x, r.y, r.z, r.w};
        uint32_t ng = 0u, ne = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (!in_range(i0 + e, c.P, pend)) continue;
          const uint32_t k = u[e] & mask;
          if (k > prefix) ng |= 1u << e;
          if (k == prefix) ne |= 1u << e;
        }
        const int rel = i0 - base;
        if (ng) atomicOr(&sm.gt[rel >> 5], ng << (rel & 31));
        if (ne) atomicOr(&sm.eq[rel >> 5], ne << (rel & 31));
      }
      __syncthreads();
    }
    // rank the equal slots in slot order; keep the first eq_left of them
    const int wpt = (words + RT - 1) / RT;  // words per thread, contiguous
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
        if (r < static_cast<unsigned>(need_total)) keep[c.P + r] = base + 32 * j + b;
        ++r;
      }
    }
    out += tot_keep;
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_rand_select(const SelectParams& p, int n_slices, cudaStream_t st) {
  const cudaError_t e = cudaFuncSetAttribute(rand_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(sizeof(RSmem)));
  if (e != cudaSuccess) return e;
  rand_select_kernel<<<n_slices, RT, sizeof(RSmem), st>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tri
