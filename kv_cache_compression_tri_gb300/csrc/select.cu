// select.cu -- per-slice budgeted top-k selection in one CTA.
//
// TriAttention paper summary, "Retention and eviction" (top-B by score) and
// Random Attention, Eq. 2 / Eq. 3 / Algorithm 1 (top-K of i.i.d. uniform
// draws, prompt forced in): keep [0, P) U top-(B-P-W) candidates U
// [n-W, n), ascending. One CTA of 1024 threads owns one slice:
//   1. candidate keys -- the order-preserving u32 of the fp32 score, or the
//      Philox-4x32-10 draw -- are staged in shared memory (up to 32768 per
//      pass, 128 KB), slot-ordered;
//   2. a 4-pass MSD radix select (8-bit digits) finds the exact threshold
//      key T and how many keys equal to T are still needed; the histogram
//      lives in shared memory and same-digit lanes are merged with
//      match.any so a warp issues one shared atomic per distinct digit; the
//      select stops early when a digit bin is taken whole;
//   3. one block-wide scan in slot order ranks the kept keys (warp ballots
//      plus one scan over (chunk, warp) counts), so the keep list comes out
//      ascending without sorting; among keys equal to T the lower slots win
//      (a second scan ranks them only when needed).
// Slices with more than 32768 candidates are processed in 32768-key
// super-chunks re-staged for every pass (scores re-read, draws recomputed).
#include <cuda_runtime.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

constexpr int NT = 1024;
constexpr int NW = NT / 32;
constexpr int KCAP = 32768;     // keys staged per super-chunk
constexpr int NCH = KCAP / NT;  // chunks of NT slots per super-chunk
constexpr size_t KEY_SMEM = KCAP * sizeof(uint32_t);

struct SliceCtx {
  int64_t s;
  int n, P, W, B;
  int lo;   // first slot of the staged range (P rounded down to 4)
  int end;  // n - W: exclusive end of the candidates
  int seq, layer, head;
};

struct Smem {
  unsigned hist[256];
  unsigned tot[NCH * NW];  // per (chunk, warp) counts, then exclusive offsets
  unsigned wsum[NW];
  unsigned total;
  int pick_digit;
  unsigned pick_above, pick_count;
  int nan_seen;
};

// Stage the keys of slots [base, base + KCAP) into skey (slot-ordered).
// Slots outside [P, end) get key 0 and are masked out by their index later.
template <bool RANDOM>
__device__ __forceinline__ void stage_keys(const SelectParams& p, const SliceCtx& c, int base,
                                           uint32_t* skey, bool& nan) {
  if (RANDOM) {
    // one Philox call yields the draws of 4 consecutive slots (base % 4 == 0)
    const uint2 key = make_uint2(static_cast<uint32_t>(p.seed), static_cast<uint32_t>(p.seed >> 32));
    const uint32_t lay = static_cast<uint32_t>(c.head + 65536 * c.layer);
    for (int g = threadIdx.x; g < KCAP / 4; g += NT) {
      const int i0 = base + 4 * g;
      uint4 r = make_uint4(0u, 0u, 0u, 0u);
      if (i0 < c.end)
        r = philox4x32_10(
            make_uint4(static_cast<uint32_t>(i0) >> 2, lay, static_cast<uint32_t>(c.seq), p.round), key);
      reinterpret_cast<uint4*>(skey)[g] = r;
    }
  } else {
    const float* row = p.scores + c.s * static_cast<int64_t>(p.n_cap);
    for (int j = threadIdx.x; j < KCAP; j += NT) {
      const int i = base + j;
      uint32_t k = 0u;
      if (i >= c.P && i < c.end) k = score_key(__ldcg(row + i), nan);
      skey[j] = k;
    }
  }
}

// Block-wide exclusive scan of sm.tot[0..count) (count <= NT), in place;
// returns the sum of all entries. Callers sync before (entries written) and
// may read sm.tot right after it returns.
__device__ unsigned block_exclusive_scan(Smem& sm, int count) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const unsigned v = (t < count) ? sm.tot[t] : 0u;
  unsigned incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    const unsigned x = sm.wsum[lane];
    unsigned xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(FULL_MASK, xi, o);
      if (lane >= o) xi += y;
    }
    sm.wsum[lane] = xi - x;  // exclusive
    if (lane == 31) sm.total = xi;
  }
  __syncthreads();
  if (t < count) sm.tot[t] = incl - v + sm.wsum[w];
  const unsigned total = sm.total;
  __syncthreads();
  return total;
}

// Flags packed one bit per chunk (bit q: slot base + q*NT + threadIdx.x).
// Writes the exclusive slot-order offset of each (chunk, warp) into
// sm.tot[q*NW + w] and returns the total.
__device__ __forceinline__ unsigned chunk_offsets(Smem& sm, uint32_t bits, int lane, int w) {
#pragma unroll
  for (int q = 0; q < NCH; ++q) {
    const unsigned b = __ballot_sync(FULL_MASK, (bits >> q) & 1u);
    if (lane == 0) sm.tot[q * NW + w] = __popc(b);
  }
  __syncthreads();
  return block_exclusive_scan(sm, NCH * NW);
}

template <bool RANDOM>
__global__ void __launch_bounds__(NT, 1) select_kernel(const __grid_constant__ SelectParams p) {
  extern __shared__ __align__(16) uint32_t skey[];
  __shared__ Smem sm;

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
  if (t == 0) sm.nan_seen = 0;
  bool nan = false;
  if (staged_once) {
    stage_keys<RANDOM>(p, c, c.lo, skey, nan);
    __syncthreads();
  }

  // ---- radix select: 4 passes of 8 bits, most significant first ----------
  uint32_t prefix = 0u, mask = 0u;
  unsigned need = static_cast<unsigned>(need_total);
  bool exact = false;
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (t < 256) sm.hist[t] = 0u;
    __syncthreads();
    for (int sc = 0; sc < n_super; ++sc) {
      const int base = c.lo + sc * KCAP;
      if (!staged_once) {
        stage_keys<RANDOM>(p, c, base, skey, nan);
        __syncthreads();
      }
      for (int q = 0; q < NCH; ++q) {
        const int j = q * NT + t;
        const int i = base + j;
        const uint32_t k = skey[j];
        const bool act = (i >= c.P) && (i < c.end) && ((k & mask) == prefix);
        const unsigned digit = act ? ((k >> shift) & 0xffu) : 256u;
        const unsigned peers = __match_any_sync(FULL_MASK, digit);
        if (act && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[digit], __popc(peers));
      }
      if (!staged_once) __syncthreads();  // skey is re-staged next
    }
    __syncthreads();
    if (w == 0) {
      // digit b with count(digits > b) < need <= count(digits >= b)
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
    __syncthreads();
    const unsigned b = static_cast<unsigned>(sm.pick_digit);
    need -= sm.pick_above;
    const unsigned cnt = sm.pick_count;
    prefix |= b << shift;
    mask |= 0xffu << shift;
    __syncthreads();  // pick_* are rewritten by the next pass
    if (cnt == need) {
      exact = true;  // every key with this prefix is kept
      break;
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
      stage_keys<RANDOM>(p, c, base, skey, nan);
      __syncthreads();
    }
    uint32_t eqb = 0u, gtb = 0u;
#pragma unroll
    for (int q = 0; q < NCH; ++q) {
      const int j = q * NT + t;
      const int i = base + j;
      const uint32_t k = skey[j] & mask;
      const bool valid = (i >= c.P) && (i < c.end);
      if (valid && k > prefix) gtb |= 1u << q;
      if (valid && k == prefix) eqb |= 1u << q;
    }
    if (!exact) {
      const unsigned total_eq = chunk_offsets(sm, eqb, lane, w);
#pragma unroll
      for (int q = 0; q < NCH; ++q) {
        const unsigned bq = __ballot_sync(FULL_MASK, (eqb >> q) & 1u);
        const unsigned rank = eq_carry + sm.tot[q * NW + w] + __popc(bq & lt_mask);
        if (((eqb >> q) & 1u) && rank >= need) eqb &= ~(1u << q);
      }
      eq_carry += total_eq;
      __syncthreads();  // sm.tot is rewritten below
    }
    const uint32_t kb = gtb | eqb;
    const unsigned total_keep = chunk_offsets(sm, kb, lane, w);
#pragma unroll
    for (int q = 0; q < NCH; ++q) {
      const unsigned bq = __ballot_sync(FULL_MASK, (kb >> q) & 1u);
      const unsigned rank = keep_carry + sm.tot[q * NW + w] + __popc(bq & lt_mask);
      if (((kb >> q) & 1u) && rank < static_cast<unsigned>(need_total))
        keep[c.P + rank] = base + q * NT + t;
    }
    keep_carry += total_keep;
    __syncthreads();
  }
  if (nan) atomicOr(&sm.nan_seen, 1);
  __syncthreads();
  if (t == 0 && sm.nan_seen) set_status(p.dev_status, TRI_DEV_NAN_SCORE);
}

template <bool RANDOM>
cudaError_t launch_one(const SelectParams& p, int n_slices, cudaStream_t st) {
  // The dynamic shared memory opt-in is a per-device function attribute;
  // setting it on every call is cheap and covers every device.
  const cudaError_t e = cudaFuncSetAttribute(select_kernel<RANDOM>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(KEY_SMEM));
  if (e != cudaSuccess) return e;
  select_kernel<RANDOM><<<n_slices, NT, KEY_SMEM, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select(const SelectParams& p, bool random, int n_slices, cudaStream_t st) {
  return random ? launch_one<true>(p, n_slices, st) : launch_one<false>(p, n_slices, st);
}

}  // namespace tri
