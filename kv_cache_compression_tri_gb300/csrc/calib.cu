// calib.cu -- offline per-(layer, KV head) query statistics.
//
// TriAttention paper summary, "Offline Calibration Procedure" and
// "Measurement via Mean Resultant Length": per band f, the centre E[q_f]
// (complex mean), the mean magnitude E|q_f| and R_f = |E q_f| / E|q_f|,
// pooling the G query heads that share a KV head.
//
// Two launches, both deterministic (fixed reduction order, no atomics):
//   calib_partial: grid (lh, split); each CTA streams a contiguous range of
//     the lh's G * n_tok pre-RoPE query rows with 16-byte loads (TPK lanes
//     per row, BPT bands per lane), accumulates sum re, sum im, sum |q_f| in
//     fp32 registers, reduces its rows through shared memory and writes one
//     partial [F][3] to the caller's scratch;
//   calib_final: grid (lh), one thread per band sums the partials in split
//     order and writes centre, mean norm and MRL.
#include <cuda_runtime.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

constexpr int CAL_T = 256;

template <typename T, int D, int STYLE>
__global__ void __launch_bounds__(CAL_T) calib_partial(const __grid_constant__ CalibParams p) {
  constexpr int F = D / 2;
  constexpr int BPT = (sizeof(T) == 2) ? 4 : 2;
  constexpr int TPK = F / BPT;
  constexpr int RPI = CAL_T / TPK;  // rows per iteration
  __shared__ float red[CAL_T * BPT * 3];

  const int lh = blockIdx.x, split = blockIdx.y;
  const int layer = lh / p.kv_heads, h = lh % p.kv_heads;
  const int64_t samples = static_cast<int64_t>(p.group) * p.n_tok;
  const int64_t a = samples * split / p.n_split, b = samples * (split + 1) / p.n_split;
  const int c = threadIdx.x % TPK, r0 = threadIdx.x / TPK;

  float sre[BPT], sim[BPT], sab[BPT];
#pragma unroll
  for (int j = 0; j < BPT; ++j) sre[j] = sim[j] = sab[j] = 0.0f;

  for (int64_t u = a + r0; u < b; u += RPI) {
    const int64_t g = u / p.n_tok, tok = u % p.n_tok;
    const int64_t qh = static_cast<int64_t>(h) * p.group + g;
    const T* row = static_cast<const T*>(p.q) + ((layer * static_cast<int64_t>(p.n_q_heads) + qh) * p.n_tok + tok) * D;
    float re[BPT], im[BPT];
    if (sizeof(T) == 2) {
      uint32_t w[4];
      if (STYLE == TRI_ROPE_INTERLEAVED) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4*>(row) + c);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
#pragma unroll
        for (int j = 0; j < 4; ++j) { re[j] = bf16_lo(w[j]); im[j] = bf16_hi(w[j]); }
      } else {
        const uint2 x = __ldcs(reinterpret_cast<const uint2*>(row) + c);
        const uint2 y = __ldcs(reinterpret_cast<const uint2*>(row + F) + c);
        re[0] = bf16_lo(x.x); re[1] = bf16_hi(x.x); re[2] = bf16_lo(x.y); re[3] = bf16_hi(x.y);
        im[0] = bf16_lo(y.x); im[1] = bf16_hi(y.x); im[2] = bf16_lo(y.y); im[3] = bf16_hi(y.y);
      }
    } else {
      if (STYLE == TRI_ROPE_INTERLEAVED) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(row) + c);
        re[0] = v.x; im[0] = v.y; re[1] = v.z; im[1] = v.w;
      } else {
        const float2 x = __ldcs(reinterpret_cast<const float2*>(row) + c);
        const float2 y = __ldcs(reinterpret_cast<const float2*>(row + F) + c);
        re[0] = x.x; re[1] = x.y; im[0] = y.x; im[1] = y.y;
      }
    }
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      sre[j] += re[j];
      sim[j] += im[j];
      sab[j] += sqrtf(fmaf(im[j], im[j], re[j] * re[j]));
    }
  }
  // rows r0 = 0..RPI-1 hold partial sums of the same bands: reduce over r0
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    red[(threadIdx.x * BPT + j) * 3 + 0] = sre[j];
    red[(threadIdx.x * BPT + j) * 3 + 1] = sim[j];
    red[(threadIdx.x * BPT + j) * 3 + 2] = sab[j];
  }
  __syncthreads();
  for (int stride = RPI / 2; stride >= 1; stride >>= 1) {
    if (r0 < stride) {
      const int other = (r0 + stride) * TPK + c;
#pragma unroll
      for (int j = 0; j < BPT * 3; ++j) red[threadIdx.x * BPT * 3 + j] += red[other * BPT * 3 + j];
    }
    __syncthreads();
  }
  if (r0 == 0) {
    float* out = p.ws + (static_cast<int64_t>(lh) * p.n_split + split) * F * 3;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      const int f = c * BPT + j;
      out[f * 3 + 0] = red[(threadIdx.x * BPT + j) * 3 + 0];
      out[f * 3 + 1] = red[(threadIdx.x * BPT + j) * 3 + 1];
      out[f * 3 + 2] = red[(threadIdx.x * BPT + j) * 3 + 2];
    }
  }
}

__global__ void calib_final(const __grid_constant__ CalibParams p, int F) {
  const int lh = blockIdx.x, f = threadIdx.x;
  if (f >= F) return;
  float sre = 0.0f, sim = 0.0f, sab = 0.0f;
  for (int sp = 0; sp < p.n_split; ++sp) {
    const float* in = p.ws + (static_cast<int64_t>(lh) * p.n_split + sp) * F * 3;
    sre += in[f * 3 + 0];
    sim += in[f * 3 + 1];
    sab += in[f * 3 + 2];
  }
  const float n = static_cast<float>(static_cast<double>(p.group) * static_cast<double>(p.n_tok));
  const float cre = sre / n, cim = sim / n, m = sab / n;
  const int64_t o = static_cast<int64_t>(lh) * F + f;
  p.center[2 * o] = cre;
  p.center[2 * o + 1] = cim;
  p.mean_norm[o] = m;
  p.mrl[o] = (m > 0.0f) ? sqrtf(cre * cre + cim * cim) / m : 0.0f;
}

template <typename T, int D>
cudaError_t launch_cal(const CalibParams& p, tri_rope_style style, int lh_count, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(lh_count), static_cast<unsigned>(p.n_split));
  if (style == TRI_ROPE_INTERLEAVED)
    calib_partial<T, D, TRI_ROPE_INTERLEAVED><<<grid, CAL_T, 0, st>>>(p);
  else
    calib_partial<T, D, TRI_ROPE_HALF><<<grid, CAL_T, 0, st>>>(p);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  calib_final<<<lh_count, 64, 0, st>>>(p, D / 2);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

// Splits per lh: enough CTAs to cover the GPU a few times over, but at least
// ~2048 rows per CTA. A pure function of the shapes (the workspace size
// query uses it too).
int calibrate_split_count(int lh_count, int64_t samples_per_lh) {
  const int64_t target_ctas = 152 * 8;
  int64_t s = (target_ctas + lh_count - 1) / lh_count;
  const int64_t max_by_rows = samples_per_lh / 2048;
  if (s > max_by_rows) s = max_by_rows;
  if (s < 1) s = 1;
  if (s > 4096) s = 4096;
  return static_cast<int>(s);
}

cudaError_t launch_calibrate(const CalibParams& p, tri_dtype dt, int head_dim,
                             tri_rope_style style, int lh_count, cudaStream_t st) {
  if (dt == TRI_BF16) {
    if (head_dim == 128) return launch_cal<uint16_t, 128>(p, style, lh_count, st);
    return launch_cal<uint16_t, 64>(p, style, lh_count, st);
  }
  if (head_dim == 128) return launch_cal<float, 128>(p, style, lh_count, st);
  return launch_cal<float, 64>(p, style, lh_count, st);
}

}  // namespace tri
