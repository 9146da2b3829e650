// select.cu -- launchers of the per-slice selection kernels (select_core.cuh).
#include <cuda_runtime.h>

#include "select_core.cuh"

namespace tri {
namespace {

template <class Src>
cudaError_t launch_src(const SelectParams& p, int n_slices, cudaStream_t st) {
  // The dynamic shared memory opt-in is a per-device function attribute;
  // setting it on every call is cheap and covers every device.
  const cudaError_t e = cudaFuncSetAttribute(select_kernel<Src>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(sizeof(SSmem)));
  if (e != cudaSuccess) return e;
  select_kernel<Src><<<n_slices, NT, sizeof(SSmem), st>>>(p);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select(const SelectParams& p, int n_slices, cudaStream_t st) {
  return launch_src<ScoreKeys>(p, n_slices, st);
}

cudaError_t launch_rand_select(const SelectParams& p, int n_slices, cudaStream_t st) {
  return launch_src<DrawKeys>(p, n_slices, st);
}

cudaError_t launch_select_union(const SelectParams& p, int n_groups, cudaStream_t st) {
  switch (p.group) {
    case 1: return launch_src<UnionKeys<1>>(p, n_groups, st);
    case 2: return launch_src<UnionKeys<2>>(p, n_groups, st);
    case 3: return launch_src<UnionKeys<3>>(p, n_groups, st);
    case 4: return launch_src<UnionKeys<4>>(p, n_groups, st);
    case 5: return launch_src<UnionKeys<5>>(p, n_groups, st);
    case 6: return launch_src<UnionKeys<6>>(p, n_groups, st);
    case 7: return launch_src<UnionKeys<7>>(p, n_groups, st);
    case 8: return launch_src<UnionKeys<8>>(p, n_groups, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_select_zmax(const SelectParams& p, int n_slices, cudaStream_t st) {
  switch (p.group) {
    case 1: return launch_src<ZMaxKeys<1>>(p, n_slices, st);
    case 2: return launch_src<ZMaxKeys<2>>(p, n_slices, st);
    case 3: return launch_src<ZMaxKeys<3>>(p, n_slices, st);
    case 4: return launch_src<ZMaxKeys<4>>(p, n_slices, st);
    case 5: return launch_src<ZMaxKeys<5>>(p, n_slices, st);
    case 6: return launch_src<ZMaxKeys<6>>(p, n_slices, st);
    case 7: return launch_src<ZMaxKeys<7>>(p, n_slices, st);
    case 8: return launch_src<ZMaxKeys<8>>(p, n_slices, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tri
