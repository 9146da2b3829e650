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
// an emission sweep flags kept slots and writes the keep list in order.
// Every sweep reads 16-byte groups of 4 slots, 8 groups in flight per thread
// (one "piece" of BS*32 slots per round), so the L2 latency is paid once per
// piece rather than once per key.
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
constexpr int BSEL_G = 8;  // 16-byte groups per thread per piece

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

// Load the keys of one piece: thread (w, lane) gets groups
// g = w*32*BSEL_G + j*32 + lane (j < BSEL_G), slots lo + 4g .. lo + 4g + 3;
// slots outside [P, end) come back invalid. row is 16-byte aligned at lo.
template <int BS>
__device__ __forceinline__ void bsel_load_piece(const float* row, int lo, int piece, int P, int end,
                                                uint32_t (&k)[BSEL_G][4], uint32_t (&valid)[BSEL_G],
                                                bool& nan) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float4 f[BSEL_G];
#pragma unroll
  for (int j = 0; j < BSEL_G; ++j) {
    const int i0 = lo + 4 * (piece * BS * BSEL_G + w * 32 * BSEL_G + j * 32 + lane);
    f[j] = (i0 < end) ? __ldcg(reinterpret_cast<const float4*>(row + i0)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int j = 0; j < BSEL_G; ++j) {
    const int i0 = lo + 4 * (piece * BS * BSEL_G + w * 32 * BSEL_G + j * 32 + lane);
    const float x[4] = {f[j].x, f[j].y, f[j].z, f[j].w};
    uint32_t v = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool ok = static_cast<unsigned>(i0 + e - P) < static_cast<unsigned>(end - P);
      k[j][e] = ok ? score_key(x[e], nan) : 0u;
      v |= static_cast<uint32_t>(ok) << e;
    }
    valid[j] = v;
  }
}

// Select for one slice. row: the slice's scores (global, already written and
// made visible; 16-byte aligned); kmin / kmax: min and max score key over the
// candidates. scratch: >= BSEL_SMEM_BYTES of shared memory. Must be called by
// all BS threads of the CTA.
template <int BS>
__device__ void block_select(const float* row, int n, int P, int W, int B, uint32_t kmin, uint32_t kmax,
                             int32_t* keep, unsigned char* scratch, int32_t* dev_status) {
  static_assert(BS % 32 == 0 && BS <= 256, "block size");
  constexpr int NWB = BS / 32;
  constexpr int PIECE = BS * BSEL_G * 4;  // slots per piece
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
  const int lo = P & ~3;
  const int n_pieces = (end - lo + PIECE - 1) / PIECE;
  uint32_t k[BSEL_G][4], valid[BSEL_G];

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
    for (int pc = 0; pc < n_pieces; ++pc) {
      bsel_load_piece<BS>(row, lo, pc, P, end, k, valid, nan);
#pragma unroll
      for (int j = 0; j < BSEL_G; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (((valid[j] >> e) & 1u) && (k[j][e] & mask) == prefix)
            atomicAdd(&sm.whist[w][(k[j][e] >> shift) & dmask], 1u);
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
    for (int pc = 0; pc < n_pieces; ++pc) {
      bsel_load_piece<BS>(row, lo, pc, P, end, k, valid, nan);
#pragma unroll
      for (int j = 0; j < BSEL_G; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (((valid[j] >> e) & 1u) && (k[j][e] & mask) == prefix) {
            const unsigned at = atomicAdd(&sm.nlist, 1u);
            if (at < static_cast<unsigned>(BSEL_LCAP)) lkey[at] = k[j][e];
          }
    }
    __syncthreads();
    const int nl = min(static_cast<int>(sm.nlist), BSEL_LCAP);
    while (!resolved) {
      for (int b = t; b < 256; b += BS) sm.hist[b] = 0u;
      __syncthreads();
      const uint32_t dmask = (1u << width) - 1u;
      for (int e = t; e < nl; e += BS) {
        const uint32_t kk = lkey[e];
        if ((kk & mask) == prefix) atomicAdd(&sm.hist[(kk >> shift) & dmask], 1u);
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

  // ---- emission, piece by piece, in slot order ------------------------------
  // Within a piece, warp w owns groups [w*32*G, (w+1)*32*G) in slot order
  // (group j*32 + lane is slot-ordered by (j, lane)); each lane holds a
  // 4-bit flag nibble per group.
  unsigned eq_carry = 0u, out = 0u;
  for (int pc = 0; pc < n_pieces; ++pc) {
    bsel_load_piece<BS>(row, lo, pc, P, end, k, valid, nan);
    uint32_t gt[BSEL_G], eq[BSEL_G];
#pragma unroll
    for (int j = 0; j < BSEL_G; ++j) {
      gt[j] = eq[j] = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t km = k[j][e] & mask;
        const uint32_t v = (valid[j] >> e) & 1u;
        gt[j] |= (v & static_cast<uint32_t>(km > prefix)) << e;
        eq[j] |= (v & static_cast<uint32_t>(km == prefix)) << e;
      }
    }
    if (!exact) {
      unsigned cnt = 0u;
#pragma unroll
      for (int j = 0; j < BSEL_G; ++j) cnt += __popc(eq[j]);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) cnt += __shfl_xor_sync(FULL_MASK, cnt, o);
      if (lane == 0) sm.wtot[w] = cnt;
      __syncthreads();
      unsigned tot;
      unsigned r = eq_carry + bsel_scan_warps<BS>(sm, w, lane, tot);
#pragma unroll
      for (int j = 0; j < BSEL_G; ++j) {
        const unsigned c = __popc(eq[j]);
        unsigned incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned y = __shfl_up_sync(FULL_MASK, incl, o);
          if (lane >= o) incl += y;
        }
        unsigned rr = r + incl - c;
        uint32_t kept = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((eq[j] >> e) & 1u) {
            if (rr < need) kept |= 1u << e;
            ++rr;
          }
        eq[j] = kept;
        r += __shfl_sync(FULL_MASK, incl, 31);
      }
      eq_carry += tot;
      __syncthreads();
    }
    unsigned cnt = 0u;
#pragma unroll
    for (int j = 0; j < BSEL_G; ++j) cnt += __popc(gt[j] | eq[j]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) cnt += __shfl_xor_sync(FULL_MASK, cnt, o);
    if (lane == 0) sm.wtot[w] = cnt;
    __syncthreads();
    unsigned tot;
    unsigned r = out + bsel_scan_warps<BS>(sm, w, lane, tot);
#pragma unroll
    for (int j = 0; j < BSEL_G; ++j) {
      const uint32_t kb = gt[j] | eq[j];
      const unsigned c = __popc(kb);
      unsigned incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += y;
      }
      unsigned rr = r + incl - c;
      const int i0 = lo + 4 * (pc * BS * BSEL_G + w * 32 * BSEL_G + j * 32 + lane);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((kb >> e) & 1u) {
          if (rr < static_cast<unsigned>(need_total)) keep[P + rr] = i0 + e;
          ++rr;
        }
      r += __shfl_sync(FULL_MASK, incl, 31);
    }
    out += tot;
    __syncthreads();
  }
  if (nan) atomicOr(&sm.nan_seen, 1);
  __syncthreads();
  if (t == 0 && sm.nan_seen) set_status(dev_status, TRI_DEV_NAN_SCORE);
}

}  // namespace tri
