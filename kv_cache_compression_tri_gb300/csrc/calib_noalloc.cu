// calib_noalloc.cu -- calibration without caller-provided scratch.
//
// tri_calibrate_centers needs a small device scratch buffer for its
// per-split partial sums, which the caller normally allocates and passes in.
// Some callers cannot do that: a plugin running inside an engine that owns
// every byte of device memory through its own pool and forbids direct driver
// allocations, or latency-critical code that must not call cudaMalloc /
// cudaFree because they can synchronise the device and stall other streams.
// tri_calibrate_centers_noalloc serves them: the scratch is a fixed-size
// array in this library's own device memory, so the call allocates nothing.
//
// The array is a file-scope __device__ variable. On the host its name is only
// a stand-in, not a device address, so every call looks up the real address
// with cudaGetSymbolAddress (a host-side query that allocates nothing) on the
// current device and passes it to the kernels. Looking it up per call, rather
// than caching it, keeps the address right after cudaDeviceReset (which loads
// the module again, possibly elsewhere) and under a different driver context
// of the same device. Every GPU that loads the library holds the array until
// the process exits.
#include <cuda_runtime.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

// 4 MiB: enough for the partial sums of e.g. 36 layers x 8 KV heads x
// head_dim 128 (about 1.1 MB with the split count the library picks).
constexpr size_t NOALLOC_SCRATCH_BYTES = TRI_CALIBRATE_NOALLOC_MAX_SCRATCH_BYTES;
static_assert(NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");

static __device__ __align__(256) float g_calib_scratch[NOALLOC_SCRATCH_BYTES / sizeof(float)];

// Device address of the scratch array in the current device's context, or
// nullptr with *err set.
float* scratch_for_current_device(cudaError_t* err) {
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_calib_scratch);
  return *err == cudaSuccess ? static_cast<float*>(p) : nullptr;
}

}  // namespace
}  // namespace tri

using namespace tri;

extern "C" {

tri_status tri_calibrate_centers_noalloc(const void* q, tri_dtype dtype, int32_t n_layers,
                                         int32_t n_q_heads, int32_t group, int32_t head_dim,
                                         int64_t n_tok, tri_rope_style style, tri_centers out,
                                         tri_stream_t stream) {
  TRI_CALL_RANGE();
  if (dtype != TRI_BF16 && dtype != TRI_F32) return TRI_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return TRI_ERR_UNSUPPORTED;
  if (style != TRI_ROPE_INTERLEAVED && style != TRI_ROPE_HALF) return TRI_ERR_INVALID_ARG;
  if (!q || (reinterpret_cast<uintptr_t>(q) % 16) != 0 || n_layers < 1 || n_q_heads < 1 ||
      group < 1 || n_q_heads % group != 0 || n_tok < 1)
    return TRI_ERR_INVALID_ARG;
  if (!out.center || !out.mean_norm || !out.mrl ||
      (reinterpret_cast<uintptr_t>(out.center) % 8) != 0 ||
      (reinterpret_cast<uintptr_t>(out.mean_norm) % 4) != 0 ||
      (reinterpret_cast<uintptr_t>(out.mrl) % 4) != 0)
    return TRI_ERR_INVALID_ARG;
  // The shapes decide the scratch size; refuse what does not fit the array.
  const size_t need = tri_calibrate_workspace_bytes(n_layers, n_q_heads, group, head_dim, n_tok);
  if (need > NOALLOC_SCRATCH_BYTES) return TRI_ERR_INVALID_ARG;

  cudaError_t err = cudaSuccess;
  float* scratch = scratch_for_current_device(&err);
  if (!scratch) return TRI_ERR_CUDA;

  CalibParams p{};
  p.q = q;
  p.ws = scratch;  // fully rewritten by the partial kernel before it is read
  p.center = out.center;
  p.mean_norm = out.mean_norm;
  p.mrl = out.mrl;
  p.n_q_heads = n_q_heads;
  p.group = group;
  p.kv_heads = n_q_heads / group;
  p.n_tok = n_tok;
  const int lh = n_layers * p.kv_heads;
  p.n_split = calibrate_split_count(lh, static_cast<int64_t>(group) * n_tok);
  const cudaError_t e = launch_calibrate(p, dtype, head_dim, style, lh, stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

}  // extern "C"
