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
constexpr int STAGES = 2;
constexpr int TILE_BYTES = 32768;
constexpr size_t RING_BYTES = static_cast<size_t>(STAGES) * TILE_BYTES;

// Control block of a CTA's tile ring of NST stages read by NW warps, placed
// after the tiles.
template <int NST, int NW = SCORE_WARPS>
struct RingCtrlN {
  uint64_t full[NST];      // the stage's tile has landed (bulk copy completion)
  unsigned consumed[NST];  // warps done with the stage's current tile
  int failed;              // a wait timed out
  int issued;              // tiles issued so far
};
using RingCtrl = RingCtrlN<STAGES>;
constexpr size_t SCORE_SMEM = RING_BYTES + (sizeof(RingCtrl) + 15) / 16 * 16;

// The ring: consecutive TILE_BYTES chunks of the CTA's rows, each filled by
// one bulk async copy (TMA, non-tensor) that completes on its stage's
// mbarrier. Warps move through it independently: a warp waits only for the
// tile it needs (bounded in wall-clock time), and the last warp to finish a
// stage refills it -- no CTA barrier per tile. The release counter's atomics,
// fenced at CTA scope, order every warp's shared-memory reads of the stage
// before the refill, which is issued after a generic-to-async proxy fence.

// Thread 0, before the CTA's first barrier.
template <int NST, int NW>
__device__ __forceinline__ void ring_init(RingCtrlN<NST, NW>& rc, int ntiles) {
#pragma unroll
  for (int st = 0; st < NST; ++st) {
    mbar_init(&rc.full[st], 1);
    rc.consumed[st] = 0u;
  }
  rc.failed = 0;
  rc.issued = min(NST, ntiles);
  mbar_init_fence();
}

template <int NST, int NW>
__device__ __forceinline__ bool ring_failed(const RingCtrlN<NST, NW>& rc) {
  return *reinterpret_cast<const volatile int*>(&rc.failed) != 0;
}

// Wait for tile t (warp-uniform result); a timeout marks the CTA failed.
template <int NST, int NW>
__device__ __forceinline__ bool ring_wait(RingCtrlN<NST, NW>& rc, int t, int lane) {
  bool ok = mbar_wait_bounded(&rc.full[t % NST], static_cast<uint32_t>((t / NST) & 1));
  ok = __all_sync(FULL_MASK, ok);
  if (!ok && lane == 0) atomicExch(&rc.failed, 1);
  return ok;
}

// A warp is done with tile t; the CTA's last warp to get there issues tile
// t + NST into the stage (issue(u) starts the copy of tile u).
template <int NST, int NW, class Issue>
__device__ __forceinline__ void ring_release(RingCtrlN<NST, NW>& rc, int t, int ntiles, int lane, const Issue& issue) {
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    if (atomicAdd(&rc.consumed[t % NST], 1u) == NW - 1) {
      atomicExch(&rc.consumed[t % NST], 0u);
      __threadfence_block();
      if (t + NST < ntiles) {
        fence_proxy_async_smem();
        issue(t + NST);
        atomicMax(&rc.issued, t + NST + 1);
      }
    }
  }
}

// After the CTA's last barrier: on a timeout, record it and let the copies
// in flight land before the shared memory is released (the last tile issued
// into each stage is the newest one there).
template <int NST, int NW>
__device__ __forceinline__ void ring_drain(RingCtrlN<NST, NW>& rc, int32_t* dev_status) {
  if (threadIdx.x == 0 && ring_failed(rc)) {
    set_status(dev_status, TRI_DEV_TIMEOUT);
    const int is = rc.issued;
    for (int u = max(0, is - NST); u < is; ++u)
      (void)mbar_wait_bounded(&rc.full[u % NST], static_cast<uint32_t>((u / NST) & 1));
  }
}

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
  static_assert(STEPS >= 4 && TPK >= STEPS && TPK <= 32, "score geometry");
};

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Where the rotation e^{i w_f (p_cur - p)} of a key comes from.
enum PosMode : int {
  POS_SLOT = 0,       // pre-RoPE keys at position = slot: one complex multiply per key advances it
  POS_EXPLICIT = 1,   // pre-RoPE keys with a position array: evaluated per key from the fixed-point phase
  POS_POST_ROPE = 2,  // post-RoPE keys carry e^{-i w_f p} already: only the constant e^{i w_f p_cur} remains
};

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
