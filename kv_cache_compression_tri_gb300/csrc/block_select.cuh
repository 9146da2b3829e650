// block_select.cuh -- top-k selection of one slice by a single CTA of BS
// threads, over fp32 scores in global memory (read through L2), for the
// fused score + select kernel (the last CTA to finish scoring a slice selects
// it while the other CTAs keep streaming keys).
//
// Same result as select_kernel (TriAttention paper summary, "Retention and
// eviction"; Random Attention, Eq. 2): keep [0, P) U top-(B-P-W) candidates
// of [P, n-W) by (score desc, slot asc) U [n-W, n), ascending; -0 equals +0,
// NaN ranks lowest (flagged). Steps: the keys' common high bits come from the
// min / max the scoring CTAs accumulated; a histogram sweep (per-warp
// private histograms) picks the bin of the first digit below them; the keys
// of that bin go to a short list on which the remaining digits are resolved;
// an emission sweep ranks kept slots with warp ballots (flags held in
// registers, 32 slots per lane per piece) and writes the keep list in order.
#pragma once

#include "tri_internal.cuh"

namespace tri {

struct BlockSelectSmem {
  unsigned whist[8][256];  // per-warp histograms (BS <= 256)
  unsigned hist[256];
  unsigned wtot[8];
  unsigned nlist;
  int pick_digit;
  unsigned pick_above, pick_count;
  int nan_seen;
};
constexpr int BSEL_LCAP = 6144;  // short-list capacity (keys)
constexpr size_t BSEL_SMEM_BYTES = sizeof(BlockSelectSmem) + BSEL_LCAP * sizeof(uint32_t);

template <int BS>
__device__ __forceinline__ unsigned bsel_scan_warps(BlockSelectSmem& sm, int w, int lane, unsigned& total) {
  constexpr int NWB = BS / 32;
  const unsigned x = (lane < NWB) ? sm.wtot[lane] : 0u;
  unsigned incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += y;
  }
  total = __shfl_sync(FULL_MASK, incl, 31);
  return __shfl_sync(FULL_MASK, incl - x, w);
}

__device__ __forceinline__ void bsel_pick(BlockSelectSmem& sm, unsigned need, int lane) {
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

// Select for one slice. row: the slice's scores (global, already written and
// made visible); kmin / kmax: min and max score key over the candidates.
// scratch: >= BSEL_SMEM_BYTES of shared memory. Must be called by all BS
// threads of the CTA.
template <int BS>
__device__ void block_select(const float* row, int n, int P, int W, int B, uint32_t kmin, uint32_t kmax,
                             int32_t* keep, unsigned char* scratch, int32_t* dev_status) {
  static_assert(BS % 32 == 0 && BS <= 256, "block size");
  constexpr int NWB = BS / 32;
  BlockSelectSmem& sm = *reinterpret_cast<BlockSelectSmem*>(scratch);
  uint32_t* lkey = reinterpret_cast<uint32_t*>(scratch + sizeof(BlockSelectSmem));
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;

  if (n <= B) {
    for (int j = t; j < B; j += BS) keep[j] = (j < n) ? j : -1;
    return;
  }
  const int end = n - W;
  const int need_total = B - P - W;
  for (int j = t; j < P; j += BS) keep[j] = j;
  for (int j = t; j < W; j += BS) keep[B - W + j] = n - W + j;
  if (need_total == 0) return;
  if (t == 0) {
    sm.nlist = 0u;
    sm.nan_seen = 0;
  }
  bool nan = false;
  auto key_at = [&](int i) -> uint32_t { return score_key(__ldcg(row + i), nan); };

  uint32_t prefix = 0u, mask = 0u;
  unsigned need = static_cast<unsigned>(need_total);
  bool exact = false, resolved = false;
  int shift = 24, width = 8;
  const uint32_t diff = kmin ^ kmax;
  if (diff == 0u) {
    prefix = kmin;
    mask = 0xffffffffu;
    resolved = true;
  } else {
    const int hb = 31 - __clz(diff);
    shift = max(hb - 7, 0);
    width = hb - shift + 1;
    mask = (hb == 31) ? 0u : ~((2u << hb) - 1u);
    prefix = kmin & mask;
  }

  // ---- histogram sweeps over all candidates (until the bin fits the list) --
  bool to_list = false;
  while (!resolved && !to_list) {
    for (int b = lane; b < 256; b += 32) sm.whist[w][b] = 0u;
    __syncwarp();
    const uint32_t dmask = (1u << width) - 1u;
#pragma unroll 4
    for (int i = P + t; i < end; i += BS) {
      const uint32_t k = key_at(i);
      if ((k & mask) == prefix) atomicAdd(&sm.whist[w][(k >> shift) & dmask], 1u);
    }
    __syncthreads();
    for (int b = t; b < 256; b += BS) {
      unsigned s = 0u;
#pragma unroll
      for (int ww = 0; ww < NWB; ++ww) s += sm.whist[ww][b];
      sm.hist[b] = s;
    }
    __syncthreads();
    if (w == 0) bsel_pick(sm, need, lane);
    __syncthreads();
    need -= sm.pick_above;
    const unsigned cnt = sm.pick_count;
    prefix |= static_cast<uint32_t>(sm.pick_digit) << shift;
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
      to_list = (cnt <= static_cast<unsigned>(BSEL_LCAP));
    }
  }

  // ---- finish on the short list -------------------------------------------
  if (!resolved) {
    for (int i0 = P; i0 < end; i0 += BS) {  // uniform trip count (ballot)
      const int i = i0 + t;
      const uint32_t k = (i < end) ? key_at(i) : 0u;
      const bool m = (i < end) && ((k & mask) == prefix);
      const unsigned bal = __ballot_sync(FULL_MASK, m);
      if (bal) {
        unsigned at = 0u;
        if (lane == 0) at = atomicAdd(&sm.nlist, static_cast<unsigned>(__popc(bal)));
        at = __shfl_sync(FULL_MASK, at, 0);
        if (m) lkey[at + __popc(bal & ((1u << lane) - 1u))] = k;
      }
    }
    __syncthreads();
    const int nl = static_cast<int>(sm.nlist);
    while (!resolved) {
      if (t < 256) sm.hist[t] = 0u;
      for (int b = t + BS; b < 256; b += BS) sm.hist[b] = 0u;
      __syncthreads();
      const uint32_t dmask = (1u << width) - 1u;
      for (int e = t; e < nl; e += BS) {
        const uint32_t k = lkey[e];
        if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & dmask], 1u);
      }
      __syncthreads();
      if (w == 0) bsel_pick(sm, need, lane);
      __syncthreads();
      need -= sm.pick_above;
      const unsigned cnt = sm.pick_count;
      prefix |= static_cast<uint32_t>(sm.pick_digit) << shift;
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

  // ---- emission: pieces of BS*32 slots; warp w takes 32 steps of 32 --------
  const unsigned lt_mask = (1u << lane) - 1u;
  constexpr int PIECE = BS * 32;
  unsigned eq_carry = 0u, out = 0u;
  for (int base = P; base < end; base += PIECE) {
    const int wb = base + w * 1024;
    uint32_t gtb = 0u, eqb = 0u;
#pragma unroll 8
    for (int q = 0; q < 32; ++q) {
      const int i = wb + q * 32 + lane;
      if (i < end) {
        const uint32_t k = key_at(i) & mask;
        gtb |= static_cast<uint32_t>(k > prefix) << q;
        eqb |= static_cast<uint32_t>(k == prefix) << q;
      }
    }
    if (!exact) {
      unsigned cnt = 0u;
#pragma unroll
      for (int q = 0; q < 32; ++q) cnt += __popc(__ballot_sync(FULL_MASK, (eqb >> q) & 1u));
      if (lane == 0) sm.wtot[w] = cnt;
      __syncthreads();
      unsigned tot;
      unsigned r = eq_carry + bsel_scan_warps<BS>(sm, w, lane, tot);
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const unsigned bq = __ballot_sync(FULL_MASK, (eqb >> q) & 1u);
        if (((eqb >> q) & 1u) && r + __popc(bq & lt_mask) >= need) eqb &= ~(1u << q);
        r += __popc(bq);
      }
      eq_carry += tot;
      __syncthreads();
    }
    const uint32_t kb = gtb | eqb;
    unsigned cnt = 0u;
#pragma unroll
    for (int q = 0; q < 32; ++q) cnt += __popc(__ballot_sync(FULL_MASK, (kb >> q) & 1u));
    if (lane == 0) sm.wtot[w] = cnt;
    __syncthreads();
    unsigned tot;
    unsigned r = out + bsel_scan_warps<BS>(sm, w, lane, tot);
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const unsigned bq = __ballot_sync(FULL_MASK, (kb >> q) & 1u);
      const unsigned rr = r + __popc(bq & lt_mask);
      if (((kb >> q) & 1u) && rr < static_cast<unsigned>(need_total)) keep[P + rr] = wb + q * 32 + lane;
      r += __popc(bq);
    }
    out += tot;
    __syncthreads();
  }
  if (nan) atomicOr(&sm.nan_seen, 1);
  __syncthreads();
  if (t == 0 && sm.nan_seen) set_status(dev_status, TRI_DEV_NAN_SCORE);
}

}  // namespace tri
