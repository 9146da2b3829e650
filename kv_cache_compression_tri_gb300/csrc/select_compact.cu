// select_compact.cu -- selection and compaction of a slice in one CTA.
//
// The compaction (compact_core.cuh) streams rows at the copy rate with little
// instruction issue; the selection (select_core.cuh) is latency-bound with
// little traffic. Running both per slice in one CTA, four CTAs per SM (64
// registers; the compaction's three-stage rings and the selection's state
// share about 49 KB), lets
// one slice's selection overlap other slices' row traffic instead of taking
// its own pass over the GPU. Semantics are exactly the two calls in sequence
// (tri_select_topk or rand_evict, then tri_compact_kv): the keep list is
// written to global memory as by the selection, then read back (ordinary
// loads) by the compaction after a CTA barrier.
#include <cuda_runtime.h>

#include "compact_core.cuh"
#include "select_core.cuh"

namespace tri {
namespace {

constexpr size_t fused_smem(bool paged) {
  const size_t c = COMPACT_SMEM + (paged ? CTAB * sizeof(int32_t) : 0);
  return c > sizeof(SSmem) ? c : sizeof(SSmem);
}

template <class Src, bool PAGED>
__global__ void __launch_bounds__(NT, 3)
    select_compact_kernel(const __grid_constant__ SelectParams ps, const __grid_constant__ CompactParams pc) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int64_t s = blockIdx.x;
  select_slice<Src>(ps, *reinterpret_cast<SSmem*>(smem), s);
  const int n = ps.n_valid[s];
  __syncthreads();  // the keep list is written; the selection's shared memory is free
  if (n > ps.n_cap || n < 0) return;  // the selection reported it and wrote no list
  compact_slice<PAGED, NT, false>(pc, CompactSmem<CSTAGES>::packed(smem), s);
}

template <class Src>
cudaError_t launch_src_compact(const SelectParams& ps, const CompactParams& pc, int n_slices, cudaStream_t st) {
  const bool paged = pc.rows.table != nullptr;
  auto kern = paged ? select_compact_kernel<Src, true> : select_compact_kernel<Src, false>;
  const size_t smem = fused_smem(paged);
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(n_slices), NT, smem, st>>>(ps, pc);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select_compact(const SelectParams& ps, const CompactParams& pc, bool random, int n_slices,
                                  cudaStream_t st) {
  if (pc.row_bytes % 16 != 0 || pc.row_bytes < 128 || pc.row_bytes > CTILE) return cudaErrorInvalidValue;
  return random ? launch_src_compact<DrawKeys>(ps, pc, n_slices, st)
                : launch_src_compact<ScoreKeys>(ps, pc, n_slices, st);
}

}  // namespace tri
