// compact.cu -- the compaction kernel on its own (compact_core.cuh) and the
// count of blocks a paged cache still uses after it.
#include <cuda_runtime.h>

#include "compact_core.cuh"

namespace tri {
namespace {

// Four paged CTAs per SM: dynamic shared memory, the static part (one
// 128-byte unit) and the 1 KB the SM reserves per CTA, within its 228 KB.
static_assert(4 * (COMPACT_SMEM + CTAB * sizeof(int32_t) + 128 + 1024) <= 228 * 1024, "paged compaction occupancy");

template <bool PAGED>
__global__ void __launch_bounds__(CT) compact_kernel(const __grid_constant__ CompactParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  compact_slice<PAGED, CT, true>(p, CompactSmem<CSTAGES>::packed(smem), blockIdx.x);
}

// One thread per sequence: blocks still holding live rows after compaction.
__global__ void blocks_used_kernel(const RowMap rows, const int32_t* __restrict__ n_valid, int32_t* out, int n_seq) {
  const int seq = blockIdx.x * blockDim.x + threadIdx.x;
  if (seq >= n_seq) return;
  int most = 0;
  for (int j = 0; j < rows.lh_count; ++j) most = max(most, n_valid[static_cast<int64_t>(seq) * rows.lh_count + j]);
  out[seq] = (most + rows.block_size - 1) / rows.block_size;
}

}  // namespace

cudaError_t launch_blocks_used(const RowMap& rows, const int32_t* n_valid, int32_t* blocks_used, int n_seq,
                               cudaStream_t st) {
  blocks_used_kernel<<<static_cast<unsigned>((n_seq + 127) / 128), 128, 0, st>>>(rows, n_valid, blocks_used, n_seq);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_compact(const CompactParams& p, int n_slices, cudaStream_t st) {
  if (p.row_bytes % 16 != 0 || p.row_bytes < 128 || p.row_bytes > CTILE) return cudaErrorInvalidValue;
  const bool paged = p.rows.table != nullptr;
  auto kern = paged ? compact_kernel<true> : compact_kernel<false>;
  const size_t smem = COMPACT_SMEM + (paged ? CTAB * sizeof(int32_t) : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(n_slices), CT, smem, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tri
