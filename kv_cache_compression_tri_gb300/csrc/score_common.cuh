// score_common.cuh -- pieces shared by the pooled and the per-query-head
// TriAttention score kernels: the CTA shape, the shared-memory tile ring and
// the decoding of one lane's 16 bytes of a key row into complex bands
// (TriAttention paper summary, "RoPE in complex form": band f pairs
// (x_2f, x_2f+1), or (x_f, x_f+d/2) in the half-split layout).
#pragma once

#include <cuda_runtime.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

constexpr int SCORE_THREADS = 256;
constexpr int SCORE_WARPS = SCORE_THREADS / 32;
constexpr int STAGES = 4;
constexpr int TILE_BYTES = 16384;
constexpr size_t SCORE_SMEM = STAGES * TILE_BYTES + STAGES * sizeof(uint64_t) + 16;

template <typename T, int D>
struct Geo {
  static constexpr int F = D / 2;
  static constexpr int BPT = (sizeof(T) == 2) ? 4 : 2;  // bands per lane (16 bytes)
  static constexpr int TPK = F / BPT;                   // lanes per key
  static constexpr int KPW = 32 / TPK;                  // keys per warp step
  static constexpr int ROW_BYTES = D * static_cast<int>(sizeof(T));
  static constexpr int TILE_ROWS = TILE_BYTES / ROW_BYTES;
  static constexpr int RPW = TILE_ROWS / SCORE_WARPS;  // rows per warp per tile
  static constexpr int STEPS = RPW / KPW;              // keys per lane per tile
  static_assert(STEPS == 4 && TPK >= STEPS && TPK <= 32, "score geometry");
};

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// 16 bytes of one key row for lane group c, from shared memory.
template <typename T, int D, int STYLE>
__device__ __forceinline__ uint4 lds_chunk(const unsigned char* row, int c) {
  if (STYLE == TRI_ROPE_INTERLEAVED) {
    return reinterpret_cast<const uint4*>(row)[c];
  } else {
    constexpr int HALF = D * static_cast<int>(sizeof(T)) / 2;
    const uint2 a = reinterpret_cast<const uint2*>(row)[c];
    const uint2 b = reinterpret_cast<const uint2*>(row + HALF)[c];
    return make_uint4(a.x, a.y, b.x, b.y);
  }
}

template <typename T, int STYLE>
__device__ __forceinline__ void decode_chunk(uint4 w, float* re, float* im) {
  if (sizeof(T) == 2) {
    if (STYLE == TRI_ROPE_INTERLEAVED) {
      re[0] = bf16_lo(w.x); im[0] = bf16_hi(w.x);
      re[1] = bf16_lo(w.y); im[1] = bf16_hi(w.y);
      re[2] = bf16_lo(w.z); im[2] = bf16_hi(w.z);
      re[3] = bf16_lo(w.w); im[3] = bf16_hi(w.w);
    } else {
      re[0] = bf16_lo(w.x); re[1] = bf16_hi(w.x); re[2] = bf16_lo(w.y); re[3] = bf16_hi(w.y);
      im[0] = bf16_lo(w.z); im[1] = bf16_hi(w.z); im[2] = bf16_lo(w.w); im[3] = bf16_hi(w.w);
    }
  } else {
    if (STYLE == TRI_ROPE_INTERLEAVED) {
      re[0] = __uint_as_float(w.x); im[0] = __uint_as_float(w.y);
      re[1] = __uint_as_float(w.z); im[1] = __uint_as_float(w.w);
    } else {
      re[0] = __uint_as_float(w.x); re[1] = __uint_as_float(w.y);
      im[0] = __uint_as_float(w.z); im[1] = __uint_as_float(w.w);
    }
  }
}

}  // namespace
}  // namespace tri
