// score.cu -- the fused TriAttention score kernel.
//
// Per cached key row i of slice s (TriAttention paper summary, section 3.4:
// "The Trigonometric Series Term", "Adaptive Weighting via Q/K
// Concentration", "Handling Multiple Future Positions"):
//   S~(i) = Re sum_f W_f e^{i w_f (p_cur - p_i)} conj(k_f) + sum_f n_f |k_f|
// with W_f = c_f G_f, G_f = (1/|D|) sum_delta e^{i w_f delta} (the offset
// average folded into one complex coefficient) and n_f = (1 - R_f) E|q_f|
// (or E|q_f| for the unweighted ablation). This equals the paper's
// (1/|D|) sum_delta [S_trig(k, age + delta) + S_norm(k)] exactly.
//
// Design (HBM-bound streaming):
//   * each warp streams a contiguous run of rows; a key row is split across
//     TPK lanes, each lane owning BPT consecutive bands and loading them with
//     one 16-byte (or two 8-byte) streaming load -- fully coalesced;
//   * per-lane band constants (W_f, n_f and the rotation state) live in
//     registers; for implicit positions the rotation e^{i w_f (p_cur - p)} is
//     advanced by one complex multiply per key (anchored once per warp run
//     from an exact fixed-point phase); for explicit positions it is
//     evaluated per key from a 64-bit fixed-point phase;
//   * U = 8 keys are loaded before any is consumed (memory-level
//     parallelism), then the U partial sums are reduced across the TPK lanes
//     with a transposed butterfly (reduce-scatter), which costs U - 1 + ...
//     shuffles instead of U * log2(TPK), and lands U consecutive scores in
//     consecutive lanes for one coalesced store.
#include <cuda_runtime.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

constexpr int SCORE_THREADS = 256;
constexpr int SCORE_WARPS = SCORE_THREADS / 32;
constexpr int U = 8;  // keys in flight per lane per batch

template <typename T, int D>
struct Layout {
  static constexpr int F = D / 2;
  static constexpr int BPT = (sizeof(T) == 2) ? 4 : 2;  // bands per lane (16 bytes)
  static constexpr int TPK = F / BPT;                   // lanes per key
  static constexpr int KPW = 32 / TPK;                  // keys per warp step
  static_assert(TPK >= U && TPK <= 32, "layout");
};

// 16 bytes of one key row for lane group c: interleaved -> one 16-byte load
// of BPT (re, im) pairs; half-split -> 8 bytes of real parts and 8 bytes of
// imaginary parts.
template <typename T, int D, int STYLE>
__device__ __forceinline__ uint4 load_chunk(const T* row, int c) {
  if (STYLE == TRI_ROPE_INTERLEAVED) {
    return __ldcs(reinterpret_cast<const uint4*>(row) + c);
  } else {
    constexpr int F = D / 2;
    const uint2 a = __ldcs(reinterpret_cast<const uint2*>(row) + c);
    const uint2 b = __ldcs(reinterpret_cast<const uint2*>(row + F) + c);
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

// Reduce-scatter of a[0..U) over the TPK lanes of one key group. On return,
// every lane holds the full sum of entry `idx` (lanes that differ only in
// the bits below TPK/U hold the same entry).
template <int TPK>
__device__ __forceinline__ float reduce_scatter(float (&a)[U], int lane, int& idx) {
  idx = 0;
  int m = TPK / 2;
#pragma unroll
  for (int v = U; v > 1; v >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < v / 2; ++j) {
      const float keep = upper ? a[j + v / 2] : a[j];
      const float send = upper ? a[j] : a[j + v / 2];
      a[j] = keep + __shfl_xor_sync(FULL_MASK, send, m);
    }
    if (upper) idx += v / 2;
    m >>= 1;
  }
  float r = a[0];
#pragma unroll
  for (int mm = TPK / U / 2; mm >= 1; mm >>= 1) r += __shfl_xor_sync(FULL_MASK, r, mm);
  return r;
}

template <typename T, int D, int STYLE, bool EXPLICIT_POS>
__global__ void __launch_bounds__(SCORE_THREADS)
    score_kernel(const __grid_constant__ ScoreParams p) {
  using LY = Layout<T, D>;
  constexpr int F = LY::F, BPT = LY::BPT, TPK = LY::TPK, KPW = LY::KPW;

  const int64_t s = blockIdx.x / p.tiles_per_slice;
  const int tile = blockIdx.x % p.tiles_per_slice;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int n = p.n_valid[s];
  if (n > p.n_cap || n < 0) {
    if (threadIdx.x == 0 && tile == 0) set_status(p.dev_status, TRI_DEV_NVALID_OVER_CAP);
    return;
  }
  const int lo = p.n_prompt, hi = n - p.n_recent;
  const int64_t rpc = static_cast<int64_t>(p.rows_per_warp) * SCORE_WARPS;
  int r0 = static_cast<int>(tile * rpc) + warp * p.rows_per_warp;
  int r1 = r0 + p.rows_per_warp;
  r0 = max(r0, lo);
  r1 = min(r1, hi);
  if (r0 >= r1) return;  // warp-uniform; no block-level sync below

  const int c = lane % TPK;   // band group of this lane
  const int kq = lane / TPK;  // key of the warp step this lane works on
  const int lh = static_cast<int>(s % p.lh_count);
  const int64_t seq = s / p.lh_count;
  const int64_t pc = p.p_cur[seq];

  // Per-lane band constants.
  float2 W[BPT], Dr[BPT], step[BPT];
  float nw[BPT];
  uint64_t nu[BPT];
#pragma unroll
  for (int b = 0; b < BPT; ++b) {
    const int f = c * BPT + b;
    const float2 cf = reinterpret_cast<const float2*>(p.center)[static_cast<int64_t>(lh) * F + f];
    const float m = p.mean_norm[static_cast<int64_t>(lh) * F + f];
    const float R = p.mrl[static_cast<int64_t>(lh) * F + f];
    nw[b] = (p.norm_mode == TRI_NORM_UNWEIGHTED) ? m : (1.0f - R) * m;
    W[b] = cmul(cf, make_float2(p.g_re[f], p.g_im[f]));
    nu[b] = p.nu[f];
    step[b] = make_float2(p.step_re[f], p.step_im[f]);
    if (!EXPLICIT_POS) Dr[b] = cmul(W[b], turns_rotation_accurate(pc - (r0 + kq), nu[b]));
  }

  const T* kbase = static_cast<const T*>(p.k) + s * p.slice_stride;
  float* out = p.scores + s * static_cast<int64_t>(p.n_cap);
  const int32_t* pos = EXPLICIT_POS ? p.pos + s * static_cast<int64_t>(p.n_cap) : nullptr;

  for (int base = r0; base < r1; base += U * KPW) {
    uint4 raw[U];
    int pp[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int row = base + u * KPW + kq;
      raw[u] = make_uint4(0u, 0u, 0u, 0u);
      pp[u] = 0;
      if (row < r1) {
        raw[u] = load_chunk<T, D, STYLE>(kbase + static_cast<int64_t>(row) * D, c);
        if (EXPLICIT_POS) pp[u] = __ldg(pos + row);
      }
    }
    float acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float re[BPT], im[BPT];
      decode_chunk<T, STYLE>(raw[u], re, im);
      float a = 0.0f;
#pragma unroll
      for (int b = 0; b < BPT; ++b) {
        float2 d;
        if (EXPLICIT_POS) {
          d = cmul(W[b], turns_rotation_fast(pc - pp[u], nu[b]));
        } else {
          d = Dr[b];
          Dr[b] = cmul(Dr[b], step[b]);
        }
        a = fmaf(d.x, re[b], a);
        a = fmaf(d.y, im[b], a);
        const float sq = fmaf(im[b], im[b], re[b] * re[b]);
        a = fmaf(nw[b] * sq, rsqrtf(fmaxf(sq, 1e-30f)), a);  // n_f |k_f|
      }
      acc[u] = a;
    }
    int idx;
    const float v = reduce_scatter<TPK>(acc, lane, idx);
    const int row = base + idx * KPW + kq;
    if ((c % (TPK / U)) == 0 && row < r1) __stcs(out + row, v);
  }
}

template <typename T, int D, int STYLE>
cudaError_t launch_typed(const ScoreParams& p, bool explicit_pos, int n_slices, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(n_slices) * p.tiles_per_slice));
  if (explicit_pos)
    score_kernel<T, D, STYLE, true><<<grid, SCORE_THREADS, 0, st>>>(p);
  else
    score_kernel<T, D, STYLE, false><<<grid, SCORE_THREADS, 0, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_style(const ScoreParams& p, tri_rope_style style, bool explicit_pos,
                         int n_slices, cudaStream_t st) {
  if (style == TRI_ROPE_INTERLEAVED)
    return launch_typed<T, D, TRI_ROPE_INTERLEAVED>(p, explicit_pos, n_slices, st);
  return launch_typed<T, D, TRI_ROPE_HALF>(p, explicit_pos, n_slices, st);
}

}  // namespace

int score_keys_per_warp_step(tri_dtype dt, int head_dim) {
  const int bpt = (dt == TRI_BF16) ? 4 : 2;
  return 32 / ((head_dim / 2) / bpt);
}

cudaError_t launch_score(const ScoreParams& p, tri_dtype dt, int head_dim, tri_rope_style style,
                         bool explicit_pos, int n_slices, cudaStream_t st) {
  if (dt == TRI_BF16) {
    if (head_dim == 128) return launch_style<uint16_t, 128>(p, style, explicit_pos, n_slices, st);
    return launch_style<uint16_t, 64>(p, style, explicit_pos, n_slices, st);
  }
  if (head_dim == 128) return launch_style<float, 128>(p, style, explicit_pos, n_slices, st);
  return launch_style<float, 64>(p, style, explicit_pos, n_slices, st);
}

}  // namespace tri
