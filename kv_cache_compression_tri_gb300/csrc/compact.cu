// compact.cu -- in-place, order-preserving K/V compaction.
//
// Random Attention, Appendix F: keep-sets are sorted chronologically and the
// KV tensors are compacted with a gather. Semantics: for j = 0, 1, ...,
// n_keep-1 in order, row j <- row keep[j]. keep is ascending with
// keep[j] >= j, so the source of destination j is never a row written by an
// earlier destination, though it may be a row that a later destination
// overwrites (keep = {1, 2, ...}).
//
// One CTA owns one slice. After validating the keep list and moving the
// positions, warp 0 moves the K rows and warp 1 the V rows, each through its
// own 4-stage ring of 8 KB shared-memory tiles:
//   * tile u (destination rows [u*TR, (u+1)*TR)) is gathered row by row with
//     bulk async copies (TMA, non-tensor) completing on the stage's mbarrier;
//   * once it has landed it is written back with ONE bulk store: past the
//     identity prefix (keep[j] == j, e.g. the protected prompt, which is
//     neither read nor written) every destination row moves, so a tile's
//     destinations are contiguous;
//   * the store of tile u overlaps the gathers of tiles u+1..u+3. This is
//     safe: every source of a later tile is >= (u+1)*TR, above every row tile
//     u writes, and tile u's own sources were read before its store was
//     issued.
// Waits on gathers are bounded in wall-clock time (TRI_DEV_TIMEOUT).
#include <cuda_runtime.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

constexpr int CT = 128;  // threads per CTA (validation, positions); warps 0-1 move rows
constexpr int CSTAGES = 4;
constexpr int CTILE = 8192;
constexpr size_t RING_BYTES = CSTAGES * CTILE;
constexpr size_t COMPACT_SMEM = 2 * RING_BYTES + 2 * CSTAGES * sizeof(uint64_t);
constexpr int POS_PER_THREAD = 8;

// Rows [first, n_keep) of one tensor of one slice, moved by one warp
// through a ring of CSTAGES tiles of CTILE bytes (see the file comment).
__device__ __forceinline__ void move_rows(char* base, unsigned char* ring, uint64_t* full, const int32_t* keep,
                                          int first, int n_keep, int rb, int lane, int32_t* dev_status) {
  const int TR = CTILE / rb;  // rows per tile
  const int u_first = first / TR;
  const int ntiles = (n_keep - 1) / TR - u_first + 1;
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < CSTAGES; ++st) mbar_init(&full[st], 1);
    mbar_init_fence();
  }
  __syncwarp();

  auto rows_of = [&](int k, int& lo_j, int& hi_j, int& t0) {
    t0 = (u_first + k) * TR;
    lo_j = max(t0, first);
    hi_j = min(t0 + TR, n_keep);
  };
  auto gather = [&](int k) {
    int lo_j, hi_j, t0;
    rows_of(k, lo_j, hi_j, t0);
    const int st = k % CSTAGES;
    if (lane == 0) mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>((hi_j - lo_j) * rb));
    __syncwarp();
    for (int j = lo_j + lane; j < hi_j; j += 32) {
      const int kj = __ldg(keep + j);
      bulk_g2s(ring + st * CTILE + (j - t0) * rb, base + static_cast<int64_t>(kj) * rb,
               static_cast<uint32_t>(rb), &full[st]);
    }
  };

  for (int k = 0; k < min(CSTAGES - 1, ntiles); ++k) gather(k);
  int k = 0;
  bool ok = true;
  for (; k < ntiles; ++k) {
    const int st = k % CSTAGES;
    ok = mbar_wait_bounded(&full[st], static_cast<uint32_t>((k / CSTAGES) & 1));
    ok = __all_sync(FULL_MASK, ok);
    if (!ok) break;
    if (lane == 0) {
      int lo_j, hi_j, t0;
      rows_of(k, lo_j, hi_j, t0);
      bulk_s2g(base + static_cast<int64_t>(lo_j) * rb, ring + st * CTILE + (lo_j - t0) * rb,
               static_cast<uint32_t>((hi_j - lo_j) * rb));
      bulk_commit();
    }
    const int kn = k + CSTAGES - 1;  // refills the stage of tile k - 1
    if (kn < ntiles) {
      if (lane == 0) bulk_wait_read<1>();  // tile k-1's store has read its stage
      __syncwarp();
      gather(kn);
    }
  }
  if (!ok && lane == 0) {
    // A gather never landed: report it and let the copies in flight finish
    // before the CTA's shared memory is released.
    set_status(dev_status, TRI_DEV_TIMEOUT);
    for (int u = k; u < min(ntiles, k + CSTAGES - 1); ++u)
      (void)mbar_wait_bounded(&full[u % CSTAGES], static_cast<uint32_t>((u / CSTAGES) & 1));
  }
  if (lane == 0) bulk_wait_all();
}

struct CSmem {
  int bad;
  int n_keep;
  int first_move;
};

__global__ void __launch_bounds__(CT) compact_kernel(const __grid_constant__ CompactParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ CSmem sm;
  const int t = threadIdx.x, lane = t & 31;
  const int64_t s = blockIdx.x;
  const int32_t* keep = p.keep + s * static_cast<int64_t>(p.budget);

  if (t == 0) {
    sm.bad = 0;
    sm.n_keep = p.budget;
    sm.first_move = p.budget;
  }
  __syncthreads();
  // Validate the keep list before touching anything: ascending, keep[j] >= j,
  // < n_cap, and -1 only as trailing padding.
#pragma unroll 4
  for (int j = t; j < p.budget; j += CT) {
    const int kj = __ldg(keep + j);
    const int prev = (j > 0) ? __ldg(keep + j - 1) : -2;
    if (kj < 0) {
      if (kj != -1) atomicOr(&sm.bad, 1);
      atomicMin(&sm.n_keep, j);
    } else {
      if (kj < j || kj >= p.n_cap || (j > 0 && (prev < 0 || prev >= kj))) atomicOr(&sm.bad, 1);
      if (kj != j) atomicMin(&sm.first_move, j);
    }
  }
  __syncthreads();
  if (sm.bad) {
    if (t == 0) set_status(p.dev_status, TRI_DEV_BAD_KEEP);
    return;
  }
  const int n_keep = sm.n_keep;
  const int first = min(sm.first_move, n_keep);

  {
    int32_t* pos_out = p.pos_out + s * static_cast<int64_t>(p.n_cap);
    const int32_t* pos_in = p.pos ? p.pos + s * static_cast<int64_t>(p.n_cap) : nullptr;
    if (pos_in == nullptr || pos_in != pos_out) {
      // distinct buffers (or positions implied by the slot): a plain gather
      for (int j = t; j < n_keep; j += CT) pos_out[j] = pos_in ? __ldg(pos_in + __ldg(keep + j)) : __ldg(keep + j);
    } else {
      // in place: read a chunk's sources, barrier, write it; sources of later
      // chunks lie above every row written so far
      for (int c0 = first; c0 < n_keep; c0 += CT * POS_PER_THREAD) {
        int32_t v[POS_PER_THREAD];
#pragma unroll
        for (int e = 0; e < POS_PER_THREAD; ++e) {
          const int j = c0 + e * CT + t;
          v[e] = (j < n_keep) ? pos_in[__ldg(keep + j)] : 0;
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < POS_PER_THREAD; ++e) {
          const int j = c0 + e * CT + t;
          if (j < n_keep) pos_out[j] = v[e];
        }
        __syncthreads();
      }
    }
    if (t == 0) p.n_valid[s] = n_keep;
  }
  if (t >= 64 || first >= n_keep) return;
  // warp 0 moves the K rows, warp 1 the V rows, each through its own ring
  const int wid = t >> 5;
  move_rows((wid == 0 ? p.k : p.v) + s * p.slice_bytes, smem + wid * RING_BYTES,
            reinterpret_cast<uint64_t*>(smem + 2 * RING_BYTES) + wid * CSTAGES, keep, first, n_keep, p.row_bytes,
            lane, p.dev_status);
}

}  // namespace

cudaError_t launch_compact(const CompactParams& p, int n_slices, cudaStream_t st) {
  if (p.row_bytes % 16 != 0 || p.row_bytes > CTILE) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(compact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(COMPACT_SMEM));
  if (e != cudaSuccess) return e;
  compact_kernel<<<static_cast<unsigned>(n_slices), CT, COMPACT_SMEM, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tri
