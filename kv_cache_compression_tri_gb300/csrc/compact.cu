// compact.cu -- in-place, order-preserving K/V compaction.
//
// Random Attention, Appendix F: keep-sets are sorted chronologically and the
// KV tensors are compacted with a gather. Semantics: for j = 0, 1, ...,
// n_keep-1 in order, row j <- row keep[j]. Because keep is ascending with
// keep[j] >= j, the source of destination j is never a row written by an
// earlier destination, but it may be a row that a LATER destination
// overwrites (keep = {1, 2, ...}). One CTA owns one (slice, tensor) and
// walks destination tiles of TR rows in ascending order:
//   read(tile t)  ->  barrier  ->  write(tile t)
// All sources of tile t are read before any row of tile t is written (the
// barrier), and every row written by tile t (< (t+1) TR) is below every
// source of later tiles (>= (t+1) TR). So the reads of tile t+1 may be
// issued before the writes of tile t: they are double-buffered in
// registers, keeping a tile of loads in flight while the previous tile
// drains. Identity rows (keep[j] == j, e.g. the protected prompt) are
// neither read nor written.
#include <cuda_runtime.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

constexpr int CT = 256;  // threads per CTA
constexpr int CU = 4;    // 16-byte items per thread per tile

struct CSmem {
  int bad;
  int n_keep;
  int first_move;
};

template <int CHUNKS>  // 16-byte chunks per row
__global__ void __launch_bounds__(CT) compact_kernel(const __grid_constant__ CompactParams p) {
  constexpr int TR = CT * CU / CHUNKS;  // rows per tile
  __shared__ CSmem sm;
  const int t = threadIdx.x;
  const int64_t s = blockIdx.x;
  const bool is_k = (blockIdx.y == 0);
  const int32_t* keep = p.keep + s * static_cast<int64_t>(p.budget);

  if (t == 0) {
    sm.bad = 0;
    sm.n_keep = p.budget;
    sm.first_move = p.budget;
  }
  __syncthreads();
  // Validate the keep list before touching anything: ascending, keep[j] >= j,
  // < n_cap, and -1 only as trailing padding.
  for (int j = t; j < p.budget; j += CT) {
    const int kj = keep[j];
    const int prev = (j > 0) ? keep[j - 1] : -2;
    if (kj < 0) {
      if (kj != -1) atomicOr(&sm.bad, 1);
      if (prev >= 0 || j == 0) atomicMin(&sm.n_keep, j);
      if (j > 0 && prev == -1) { /* padding continues */ }
    } else {
      if (kj < j || kj >= p.n_cap || (j > 0 && (prev < 0 || prev >= kj))) atomicOr(&sm.bad, 1);
      if (kj != j) atomicMin(&sm.first_move, j);
    }
  }
  __syncthreads();
  if (sm.bad) {
    if (t == 0 && is_k) set_status(p.dev_status, TRI_DEV_BAD_KEEP);
    return;
  }
  const int n_keep = sm.n_keep;
  const int first = min(sm.first_move, n_keep);

  char* base = (is_k ? p.k : p.v) + s * p.slice_bytes;
  const int64_t rb = p.row_bytes;
  int32_t* pos_out = p.pos_out + s * static_cast<int64_t>(p.n_cap);
  const int32_t* pos_in = p.pos ? p.pos + s * static_cast<int64_t>(p.n_cap) : nullptr;
  const bool pos_in_place = (pos_in != nullptr) && (pos_in == pos_out);

  // Positions that are not moved in place: a plain gather (or the slot index).
  if (is_k && !pos_in_place) {
    for (int j = t; j < n_keep; j += CT) pos_out[j] = pos_in ? pos_in[keep[j]] : keep[j];
  }

  uint4 A[CU], Bv[CU];
  int32_t pa = 0, pb = 0;
  auto read_tile = [&](int t0, uint4 (&buf)[CU], int32_t& pbuf) {
#pragma unroll
    for (int u = 0; u < CU; ++u) {
      const int item = t + u * CT;
      const int j = t0 + item / CHUNKS;
      const int ch = item % CHUNKS;
      if (j < n_keep) {
        const int kj = keep[j];
        if (kj != j)
          buf[u] = __ldcs(reinterpret_cast<const uint4*>(base + kj * rb) + ch);
      }
    }
    if (is_k && pos_in_place && t < TR) {
      const int j = t0 + t;
      if (j < n_keep) {
        const int kj = keep[j];
        if (kj != j) pbuf = pos_in[kj];
      }
    }
  };
  auto write_tile = [&](int t0, const uint4 (&buf)[CU], int32_t pbuf) {
#pragma unroll
    for (int u = 0; u < CU; ++u) {
      const int item = t + u * CT;
      const int j = t0 + item / CHUNKS;
      const int ch = item % CHUNKS;
      if (j < n_keep && keep[j] != j)
        __stcs(reinterpret_cast<uint4*>(base + j * rb) + ch, buf[u]);
    }
    if (is_k && pos_in_place && t < TR) {
      const int j = t0 + t;
      if (j < n_keep && keep[j] != j) pos_out[j] = pbuf;
    }
  };

  int t0 = (first / TR) * TR;
  if (t0 < n_keep) {
    read_tile(t0, A, pa);
    for (;;) {
      __syncthreads();  // all reads of tile t0 are performed before its writes
      if (t0 + TR < n_keep) read_tile(t0 + TR, Bv, pb);
      write_tile(t0, A, pa);
      t0 += TR;
      if (t0 >= n_keep) break;
      __syncthreads();
      if (t0 + TR < n_keep) read_tile(t0 + TR, A, pa);
      write_tile(t0, Bv, pb);
      t0 += TR;
      if (t0 >= n_keep) break;
    }
  }
  if (is_k && t == 0) p.n_valid[s] = n_keep;
}

}  // namespace

cudaError_t launch_compact(const CompactParams& p, int n_slices, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(n_slices), 2);
  switch (p.row_bytes / 16) {
    case 8:
      compact_kernel<8><<<grid, CT, 0, st>>>(p);
      break;
    case 16:
      compact_kernel<16><<<grid, CT, 0, st>>>(p);
      break;
    case 32:
      compact_kernel<32><<<grid, CT, 0, st>>>(p);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  note_launch();
  return cudaGetLastError();
}

}  // namespace tri
