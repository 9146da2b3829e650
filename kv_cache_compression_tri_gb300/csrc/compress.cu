// compress.cu -- one compression event of slices that fit one score CTA
// (tri_compress when n_cap is at most the score kernel's rows per CTA):
// score, selection and compaction of a slice by one CTA, in one launch.
//
// The CTA scores its slice's candidates (score_core.cuh, the score kernel's
// own CTA body), selects the slice from the scores it has just written
// (select_core.cuh; they are still in L2), then compacts it from the keep
// list it has just written (compact_core.cuh). Three CTAs share an SM, so
// one slice's latency-bound selection overlaps other slices' score and row
// traffic instead of taking a pass over the GPU of its own. Semantics are
// exactly tri_score on rows [P, n - W), tri_select_topk and tri_compact_kv in
// sequence.
#include <cuda_runtime.h>

#include "compact_core.cuh"
#include "score_core.cuh"
#include "select_core.cuh"

namespace tri {
namespace {

// The selection's state and the compaction's rings overlay the score ring's
// tiles only; the compaction's mbarriers and a paged cache's table copy come
// after the score ring's control block, so no barrier object is repurposed.
// The three phases use one CTA shape. Three CTAs share an SM (registers), so
// the compaction takes four ring stages per tensor here (the standalone
// kernel, at four CTAs per SM, has three): more bytes in flight while the
// SM's other CTAs score or select.
constexpr int FUSED_CSTAGES = 4;
using FusedCompactSmem = CompactSmem<FUSED_CSTAGES>;
static_assert(sizeof(SSmem) <= RING_BYTES, "selection state must fit in the score ring's tiles");
static_assert(2 * FusedCompactSmem::RING <= RING_BYTES, "compaction rings must fit in the score ring's tiles");
static_assert(SCORE_SMEM % 16 == 0, "compaction mbarriers after the score ring's control block");
static_assert(NT == SCORE_THREADS, "one CTA shape for the score and the selection");

constexpr size_t fused_smem(bool paged) {
  return SCORE_SMEM + FusedCompactSmem::BARS + (paged ? CTAB * sizeof(int32_t) : 0);
}

template <typename T, int D, int STYLE, int PM, bool PAGED>
__global__ void __launch_bounds__(SCORE_THREADS, 3)
    compress_slice_kernel(const __grid_constant__ ScoreParams p, const __grid_constant__ SelectParams ps,
                          const __grid_constant__ CompactParams pc) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int64_t s = blockIdx.x;
  score_cta<T, D, STYLE, PM, PAGED, false>(p, smem, s, 0);
  __syncthreads();  // the slice's scores are written (global memory, read back through L2 below)
  select_slice<ScoreKeys>(ps, *reinterpret_cast<SSmem*>(smem), s);
  const int n = ps.n_valid[s];
  __syncthreads();  // the keep list is written; the selection's shared memory is free
  if (n > ps.n_cap || n < 0) return;  // the selection reported it and wrote no list
  const FusedCompactSmem cs{smem, reinterpret_cast<uint64_t*>(smem + SCORE_SMEM),
                            reinterpret_cast<int32_t*>(smem + SCORE_SMEM + FusedCompactSmem::BARS)};
  compact_slice<PAGED, SCORE_THREADS, false, FUSED_CSTAGES>(pc, cs, s);
}

template <typename T, int D, int STYLE, int PM>
cudaError_t launch_one(const ScoreParams& p, const SelectParams& ps, const CompactParams& pc, int n_slices,
                       cudaStream_t st) {
  const bool paged = p.rows.table != nullptr;
  auto kern = paged ? compress_slice_kernel<T, D, STYLE, PM, true> : compress_slice_kernel<T, D, STYLE, PM, false>;
  const size_t smem = fused_smem(paged);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(n_slices), SCORE_THREADS, smem, st>>>(p, ps, pc);
  note_launch();
  return cudaGetLastError();
}

template <typename T, int D, int STYLE>
cudaError_t launch_pm(const ScoreParams& p, const SelectParams& ps, const CompactParams& pc, int pm, int n_slices,
                      cudaStream_t st) {
  if (pm == POS_POST_ROPE) return launch_one<T, D, STYLE, POS_POST_ROPE>(p, ps, pc, n_slices, st);
  if (pm == POS_EXPLICIT) return launch_one<T, D, STYLE, POS_EXPLICIT>(p, ps, pc, n_slices, st);
  return launch_one<T, D, STYLE, POS_SLOT>(p, ps, pc, n_slices, st);
}

template <typename T, int D>
cudaError_t launch_style(const ScoreParams& p, const SelectParams& ps, const CompactParams& pc,
                         tri_rope_style style, int pm, int n_slices, cudaStream_t st) {
  if (style == TRI_ROPE_INTERLEAVED) return launch_pm<T, D, TRI_ROPE_INTERLEAVED>(p, ps, pc, pm, n_slices, st);
  return launch_pm<T, D, TRI_ROPE_HALF>(p, ps, pc, pm, n_slices, st);
}

}  // namespace

cudaError_t launch_compress_slices(const ScoreParams& p, const SelectParams& ps, const CompactParams& pc,
                                   tri_dtype dt, int head_dim, tri_rope_style style, int pos_mode, int n_slices,
                                   cudaStream_t st) {
  if (p.tiles_per_slice != 1) return cudaErrorInvalidValue;  // a slice must fit one score CTA
  if (pc.row_bytes % 16 != 0 || pc.row_bytes < 128 || pc.row_bytes > CTILE) return cudaErrorInvalidValue;
  if (dt == TRI_BF16) {
    if (head_dim == 128) return launch_style<uint16_t, 128>(p, ps, pc, style, pos_mode, n_slices, st);
    return launch_style<uint16_t, 64>(p, ps, pc, style, pos_mode, n_slices, st);
  }
  if (head_dim == 128) return launch_style<float, 128>(p, ps, pc, style, pos_mode, n_slices, st);
  return launch_style<float, 64>(p, ps, pc, style, pos_mode, n_slices, st);
}

}  // namespace tri
