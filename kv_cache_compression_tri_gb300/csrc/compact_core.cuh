// compact_core.cuh -- in-place, order-preserving K/V compaction of one slice
// by one CTA (compact.cu launches it alone, select_compact.cu after the
// slice's selection in the same CTA).
//
// Random Attention, Appendix F: each head's kept slots, put back in time
// order, are gathered to the front of its K and V. Semantics: for j = 0, 1, ...,
// n_keep-1 in order, row j <- row keep[j]. keep is ascending with
// keep[j] >= j, so the source of destination j is never a row written by an
// earlier destination, though it may be a row that a later destination
// overwrites (keep = {1, 2, ...}).
//
// One CTA owns one slice. After validating the keep list, warp 0 moves the K
// rows and warp 1 the V rows, each through its own 3-stage ring of 8 KB
// shared-memory tiles, while warps 2-3 move the positions:
//   * tile u (destination rows [u*TR, (u+1)*TR)) is gathered with bulk async
//     copies (TMA, non-tensor) completing on the stage's mbarrier, one per
//     run of rows whose sources are adjacent in memory;
//   * once it has landed it is written back with ONE bulk store: past the
//     identity prefix (keep[j] == j, e.g. the protected prompt, which is
//     neither read nor written) every destination row moves, so a tile's
//     destinations are contiguous;
//   * the store of tile u overlaps the gathers of the following tiles. This is
//     safe: every source of a later tile is >= (u+1)*TR, above every row tile
//     u writes, and tile u's own sources were read before its store was
//     issued.
// A paged cache (block table per sequence) moves the same logical rows; the
// physical rows come from the table, and a tile's store is split where its
// destinations cross a block boundary. Waits on gathers are bounded in
// wall-clock time (TRI_DEV_TIMEOUT).
#pragma once

#include <cuda_runtime.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

constexpr int CT = 128;  // threads per CTA: warps 0-1 move K/V rows, warps 2-3 positions
constexpr int CSTAGES = 3;
constexpr int CTILE = 8192;
constexpr size_t CRING_BYTES = CSTAGES * CTILE;
constexpr size_t COMPACT_SMEM = 2 * CRING_BYTES + 2 * CSTAGES * sizeof(uint64_t);

// Where a compaction CTA keeps its shared state: the K and V rings (NST
// tiles each, V's right after K's), 2 NST mbarriers, and for a paged cache
// the copy of CTAB table entries.
template <int NST>
struct CompactSmem {
  unsigned char* rings;
  uint64_t* bars;
  int32_t* ctab;
  static constexpr size_t RING = static_cast<size_t>(NST) * CTILE;  // one tensor's
  static constexpr size_t BARS = 2 * NST * sizeof(uint64_t);
  // the standalone kernels' layout: rings, then mbarriers, then the table
  __device__ static CompactSmem packed(unsigned char* smem) {
    return {smem, reinterpret_cast<uint64_t*>(smem + 2 * RING), reinterpret_cast<int32_t*>(smem + 2 * RING + BARS)};
  }
};
// Paged: table entries cached in shared memory, from the block of the first
// row that moves (later ones are read from global). 2000 entries keep a paged
// compaction CTA within a quarter of the SM's 228 KB (with the 1 KB each CTA
// reserves), so four run per SM as in the contiguous case; 2048 would drop it
// to three.
constexpr int CTAB = 2000;
constexpr int POS_PER_THREAD = 8;

// A keep entry: through the read-only cache when the list is read-only for
// the whole kernel, else an ordinary load (the fused kernel writes it first).
template <bool RO>
__device__ __forceinline__ int keep_at(const int32_t* keep, int j) {
  return RO ? __ldg(keep + j) : keep[j];
}

// Rows [first, n_keep) of one tensor of one slice, moved by one warp
// through a ring of NST tiles of CTILE bytes (see the file comment).
// Row r of the slice is at pool + rows.row(sbase, trow, r).
template <bool PAGED, bool RO, int NST>
__device__ __forceinline__ void move_rows(char* pool, const RowMap& rows, int64_t sbase, const int32_t* trow,
                                          const int32_t* ctab, int cb0, unsigned char* ring, uint64_t* full,
                                          const int32_t* keep, int first, int n_keep, int rb, int lane,
                                          int32_t* dev_status) {
  // paged row offsets (rows >= first): entries of blocks cb0 .. cb0 + CTAB - 1
  // from the copy in shared memory, later ones from the table
  auto paged_row = [&](int r) {
    const int i = (r >> rows.block_shift) - cb0;
    const int64_t blk = (i < CTAB) ? ctab[i] : __ldg(trow + (r >> rows.block_shift));
    return sbase + blk * rows.block_bytes + static_cast<int64_t>(r & (rows.block_size - 1)) * rows.row_bytes;
  };
  const int TR = CTILE / rb;  // rows per tile
  const int u_first = first / TR;
  const int ntiles = (n_keep - 1) / TR - u_first + 1;
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < NST; ++st) mbar_init(&full[st], 1);
    mbar_init_fence();
  }
  __syncwarp();

  auto rows_of = [&](int k, int& lo_j, int& hi_j, int& t0) {
    t0 = (u_first + k) * TR;
    lo_j = max(t0, first);
    hi_j = min(t0 + TR, n_keep);
  };
  // Each lane copies rows lo_j + lane + 32 r of a tile (r < RPL); the byte
  // offsets of their sources (keep entry, and block for a paged cache) are
  // resolved one tile ahead so no gather waits on them.
  constexpr int RPL = CTILE / 128 / 32;  // most rows a lane copies per tile (2)
  int64_t knext[RPL];
  auto load_keep = [&](int k, int64_t (&kv)[RPL]) {
    int lo_j, hi_j, t0;
    rows_of(k, lo_j, hi_j, t0);
#pragma unroll
    for (int r = 0; r < RPL; ++r) {
      const int j = lo_j + lane + 32 * r;
      // (paged: a row that moves, so that its table entry is in the cache's range)
      const int src = (k < ntiles && j < hi_j) ? keep_at<RO>(keep, j) : (PAGED ? first : 0);
      kv[r] = PAGED ? paged_row(src) : sbase + static_cast<int64_t>(src) * rb;
    }
  };
  auto gather = [&](int k, const int64_t (&kv)[RPL]) {
    int lo_j, hi_j, t0;
    rows_of(k, lo_j, hi_j, t0);
    const int st = k % NST;
    if (lane == 0) mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>((hi_j - lo_j) * rb));
    __syncwarp();
    // Rows lo_j + 32 r + (0..31) sit in lanes 0..31. A row whose source
    // directly follows the previous lane's source in memory continues that
    // lane's run; each run is one bulk copy (kept rows are often adjacent
    // when a large share of the candidates survives).
#pragma unroll
    for (int r = 0; r < RPL; ++r) {
      const int j = lo_j + lane + 32 * r;
      const bool valid = j < hi_j;
      const int64_t prev = __shfl_up_sync(FULL_MASK, kv[r], 1);
      const bool cont = valid && lane > 0 && kv[r] == prev + rb;
      const unsigned runs = __ballot_sync(FULL_MASK, cont);
      if (valid && !cont) {
        const unsigned after = (lane == 31) ? 0u : (runs >> (lane + 1));  // continuations after this lane
        const int len = 1 + (__ffs(~after) - 1);
        bulk_g2s(ring + st * CTILE + (j - t0) * rb, pool + kv[r], static_cast<uint32_t>(len * rb), &full[st]);
      }
    }
  };

  for (int k = 0; k < min(NST - 1, ntiles); ++k) {
    int64_t kv[RPL];
    load_keep(k, kv);
    gather(k, kv);
  }
  load_keep(NST - 1, knext);
  int k = 0;
  bool ok = true;
  for (; k < ntiles; ++k) {
    const int st = k % NST;
    ok = mbar_wait_bounded(&full[st], static_cast<uint32_t>((k / NST) & 1));
    ok = __all_sync(FULL_MASK, ok);
    if (!ok) break;
    if (lane == 0) {
      // the tile's destinations are consecutive rows: one store per run of
      // them that is contiguous in memory (all of them, or per block)
      int lo_j, hi_j, t0;
      rows_of(k, lo_j, hi_j, t0);
      if (!PAGED) {
        bulk_s2g(pool + sbase + static_cast<int64_t>(lo_j) * rb, ring + st * CTILE + (lo_j - t0) * rb,
                 static_cast<uint32_t>((hi_j - lo_j) * rb));
      } else {
        for (int j = lo_j; j < hi_j;) {
          const int run = rows.run(j, hi_j - j);
          bulk_s2g(pool + paged_row(j), ring + st * CTILE + (j - t0) * rb, static_cast<uint32_t>(run * rb));
          j += run;
        }
      }
      bulk_commit();
    }
    const int kn = k + NST - 1;  // refills the stage of tile k - 1
    if (kn < ntiles) {
      int64_t kv[RPL];
#pragma unroll
      for (int r = 0; r < RPL; ++r) kv[r] = knext[r];
      load_keep(kn + 1, knext);
      if (lane == 0) bulk_wait_read<1>();  // tile k-1's store has read its stage
      __syncwarp();
      gather(kn, kv);
    }
  }
  if (!ok && lane == 0) {
    // A gather never landed: report it and let the copies in flight finish
    // before the CTA's shared memory is released.
    set_status(dev_status, TRI_DEV_TIMEOUT);
    for (int u = k; u < min(ntiles, k + NST - 1); ++u)
      (void)mbar_wait_bounded(&full[u % NST], static_cast<uint32_t>((u / NST) & 1));
  }
  if (lane == 0) bulk_wait_all();
}

struct CSmem {
  int bad;
  int n_keep;
  int first_move;
  int last_src;
  int bad_block;
};

// Slice s, by a CTA of NTH threads (NTH >= 128): warps 0 and 1 move the K
// and V rows through rings of NST tiles, the other warps the positions.
// RO: the keep list is read-only for the whole kernel (else it was written
// earlier in the same kernel).
template <bool PAGED, int NTH, bool RO, int NST = CSTAGES>
__device__ __forceinline__ void compact_slice(const CompactParams& p, const CompactSmem<NST>& cs, int64_t s) {
  static_assert(NTH >= 128 && NTH % 32 == 0, "compaction CTA");
  __shared__ CSmem sm;
  const int t = threadIdx.x, lane = t & 31;
  const int32_t* keep = p.keep + s * static_cast<int64_t>(p.budget);

  if (t == 0) {
    sm.bad = 0;
    sm.n_keep = p.budget;
    sm.first_move = p.budget;
    sm.last_src = -1;
  }
  __syncthreads();
  // Validate the keep list before touching anything: ascending, keep[j] >= j,
  // < n_cap, and -1 only as trailing padding. Each thread checks runs of 4
  // entries (one 16-byte load when the list is 16-byte aligned).
  const bool vec = (p.budget % 4 == 0) && ((reinterpret_cast<uintptr_t>(keep) & 15) == 0);
  int bad = 0, nk = p.budget, fm = p.budget, ls = -1;
  for (int j0 = 4 * t; j0 < p.budget; j0 += 4 * NTH) {
    int v[4];
    if (vec) {
      const int4* q4 = reinterpret_cast<const int4*>(keep + j0);
      const int4 q = RO ? __ldg(q4) : *q4;
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = (j0 + e < p.budget) ? keep_at<RO>(keep, j0 + e) : -1;
    }
    int prev = (j0 > 0) ? keep_at<RO>(keep, j0 - 1) : -2;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = j0 + e;
      if (j >= p.budget) break;
      const int kj = v[e];
      if (kj < 0) {
        bad |= (kj != -1);
        nk = min(nk, j);
      } else {
        bad |= (kj < j || kj >= p.n_cap || (j > 0 && (prev < 0 || prev >= kj)));
        if (kj != j) fm = min(fm, j);
        ls = max(ls, kj);
      }
      prev = kj;
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    bad |= __shfl_xor_sync(FULL_MASK, bad, o);
    nk = min(nk, __shfl_xor_sync(FULL_MASK, nk, o));
    fm = min(fm, __shfl_xor_sync(FULL_MASK, fm, o));
    ls = max(ls, __shfl_xor_sync(FULL_MASK, ls, o));
  }
  if (lane == 0) {
    if (bad) atomicOr(&sm.bad, 1);
    atomicMin(&sm.n_keep, nk);
    atomicMin(&sm.first_move, fm);
    atomicMax(&sm.last_src, ls);
  }
  __syncthreads();
  if (sm.bad) {
    if (t == 0) set_status(p.dev_status, TRI_DEV_BAD_KEEP);
    return;
  }
  const int n_keep = sm.n_keep;
  const int first = min(sm.first_move, n_keep);
  // a paged cache: every block the move reads or writes must be in the pool
  const int64_t sbase = p.rows.slice_base(s);
  const int32_t* trow = p.rows.seq_table(s);
  const int r1 = max(sm.last_src + 1, n_keep);
  // rows below `first` are neither read nor written, but every entry up to
  // r1 is checked; the cache holds the entries from first's block on
  const int cb0 = first >> p.rows.block_shift;
  int32_t* ctab = PAGED ? cs.ctab : nullptr;
  if (PAGED && !p.rows.blocks_ok(trow, 0, r1, &sm.bad_block, ctab, cb0, CTAB)) {
    if (t == 0) set_status(p.dev_status, TRI_DEV_BAD_BLOCK);
    return;
  }

  const int wid = t >> 5;
  if (wid < 2) {
    // warp 0 moves the K rows, warp 1 the V rows, each through its own ring
    if (first < n_keep)
      move_rows<PAGED, RO, NST>(wid == 0 ? p.k : p.v, p.rows, sbase, trow, ctab, cb0, cs.rings + wid * cs.RING,
                                cs.bars + wid * NST, keep, first, n_keep, p.row_bytes, lane, p.dev_status);
    return;
  }
  // the other warps move the positions meanwhile
  const int pt = t - 64;  // 0 .. PT-1
  constexpr int PT = NTH - 64;
  int32_t* pos_out = p.pos_out + s * static_cast<int64_t>(p.n_cap);
  const int32_t* pos_in = p.pos ? p.pos + s * static_cast<int64_t>(p.n_cap) : nullptr;
  if (pos_in == nullptr || pos_in != pos_out) {
    // distinct buffers (or positions implied by the slot): a plain gather
    for (int j = pt; j < n_keep; j += PT) {
      const int kj = keep_at<RO>(keep, j);
      pos_out[j] = pos_in ? __ldg(pos_in + kj) : kj;
    }
  } else {
    // in place: read a chunk's sources, barrier, write it; sources of later
    // chunks lie above every row written so far
    for (int c0 = first; c0 < n_keep; c0 += PT * POS_PER_THREAD) {
      int32_t v[POS_PER_THREAD];
#pragma unroll
      for (int e = 0; e < POS_PER_THREAD; ++e) {
        const int j = c0 + e * PT + pt;
        v[e] = (j < n_keep) ? pos_in[keep_at<RO>(keep, j)] : 0;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(PT) : "memory");
#pragma unroll
      for (int e = 0; e < POS_PER_THREAD; ++e) {
        const int j = c0 + e * PT + pt;
        if (j < n_keep) pos_out[j] = v[e];
      }
      asm volatile("bar.sync 1, %0;" ::"n"(PT) : "memory");
    }
  }
  if (pt == 0) p.n_valid[s] = n_keep;
}

}  // namespace
}  // namespace tri
