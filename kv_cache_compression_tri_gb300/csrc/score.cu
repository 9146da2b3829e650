// score.cu -- the score kernel (score_core.cuh: one CTA per run of a slice's
// rows) and its launchers.
#include <cuda_runtime.h>

#include "score_core.cuh"

namespace tri {
namespace {

template <typename T, int D, int STYLE, int PM, bool PAGED>
__global__ void __launch_bounds__(SCORE_THREADS, 3)
    score_kernel(const __grid_constant__ ScoreParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  score_cta<T, D, STYLE, PM, PAGED, true>(p, smem, blockIdx.x / p.tiles_per_slice,
                                          static_cast<int>(blockIdx.x % p.tiles_per_slice));
}

template <typename T, int D, int STYLE, int PM>
cudaError_t launch_one(const ScoreParams& p, int n_slices, cudaStream_t st) {
  auto kern = p.rows.table ? score_kernel<T, D, STYLE, PM, true> : score_kernel<T, D, STYLE, PM, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SCORE_SMEM));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(n_slices) * p.tiles_per_slice));
  kern<<<grid, SCORE_THREADS, SCORE_SMEM, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

template <typename T, int D, int STYLE>
cudaError_t launch_pm(const ScoreParams& p, int pm, int n_slices, cudaStream_t st) {
  if (pm == POS_POST_ROPE) return launch_one<T, D, STYLE, POS_POST_ROPE>(p, n_slices, st);
  if (pm == POS_EXPLICIT) return launch_one<T, D, STYLE, POS_EXPLICIT>(p, n_slices, st);
  return launch_one<T, D, STYLE, POS_SLOT>(p, n_slices, st);
}

template <typename T, int D>
cudaError_t launch_style(const ScoreParams& p, tri_rope_style style, int pm, int n_slices, cudaStream_t st) {
  if (style == TRI_ROPE_INTERLEAVED) return launch_pm<T, D, TRI_ROPE_INTERLEAVED>(p, pm, n_slices, st);
  return launch_pm<T, D, TRI_ROPE_HALF>(p, pm, n_slices, st);
}

template <typename T, int D>
ScoreGeometry geo() {
  using G = Geo<T, D>;
  return ScoreGeometry{G::KPW, G::TILE_ROWS - G::RPW, G::TILE_ROWS};
}

}  // namespace

ScoreGeometry score_geometry(tri_dtype dt, int head_dim) {
  if (dt == TRI_BF16) return head_dim == 128 ? geo<uint16_t, 128>() : geo<uint16_t, 64>();
  return head_dim == 128 ? geo<float, 128>() : geo<float, 64>();
}

cudaError_t launch_score(const ScoreParams& p, tri_dtype dt, int head_dim, tri_rope_style style,
                         int pos_mode, int n_slices, cudaStream_t st) {
  if (dt == TRI_BF16) {
    if (head_dim == 128) return launch_style<uint16_t, 128>(p, style, pos_mode, n_slices, st);
    return launch_style<uint16_t, 64>(p, style, pos_mode, n_slices, st);
  }
  if (head_dim == 128) return launch_style<float, 128>(p, style, pos_mode, n_slices, st);
  return launch_style<float, 64>(p, style, pos_mode, n_slices, st);
}

}  // namespace tri
