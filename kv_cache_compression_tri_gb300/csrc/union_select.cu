// union_select.cu -- the group pass of union-based selection across heads.
//
// TriAttention blog, "eviction (union-based selection)": the KV heads that
// share one keep list (here the H KV heads of one (seq, layer)) each pick
// their own top candidates; the union of the picks is kept first, ranked by a
// combined score, and topped up by the combined score when it is smaller
// than the budget. The picks come from the ordinary per-slice selection
// (select.cu, budget P + W + k_head); the final ranking is the grouped key
// source of select.cu. Between them:
//   * slice_stats_kernel, one CTA per slice: the mean and standard deviation
//     of the slice's scores over its valid rows (two passes over the slice:
//     the mean, then the centred squares), which turn the scores into the
//     z-scores of the combined score max_h z_h (TriAttention paper summary,
//     "Handling Grouped-Query Attention": normalise, then take the maximum);
//   * union_prep_kernel, one CTA per group: the union of the heads' picks as
//     a bitmap over the slots, and its size.
// The heads of a group must hold the same number of rows (their keep list is
// shared); a group that does not sets TRI_DEV_GROUP_NVALID and keeps nothing
// from the union.
#include <cuda_runtime.h>

#include <math.h>

#include "tri_internal.cuh"

namespace tri {
namespace {

constexpr int UT = 256;
constexpr int UW = UT / 32;

// Sum over the CTA in fp64, fixed order (lanes, then warps); every thread
// gets the result.
__device__ __forceinline__ double block_sum(double v, double* sred) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  if (lane == 0) sred[w] = v;
  __syncthreads();
  double tot = 0.0;
#pragma unroll
  for (int j = 0; j < UW; ++j) tot += sred[j];
  __syncthreads();  // sred is reused by the next call
  return tot;
}

__global__ void __launch_bounds__(UT) union_prep_kernel(const __grid_constant__ UnionPrepParams q) {
  extern __shared__ __align__(16) uint32_t sbits[];  // [member_words]
  __shared__ double sred[UW];
  __shared__ int sbad;
  const int t = threadIdx.x;
  const int64_t g = blockIdx.x;
  const int64_t s0 = g * q.group;
  uint32_t* member = q.member + g * q.member_words;

  if (t == 0) sbad = 0;
  __syncthreads();
  const int n = q.n_valid[s0];
  if (t < q.group && q.n_valid[s0 + t] != n) atomicExch(&sbad, 1);
  for (int j = t; j < q.member_words; j += UT) sbits[j] = 0u;
  __syncthreads();
  if (sbad || n < 0 || n > q.n_cap) {
    if (t == 0) {
      if (sbad) set_status(q.dev_status, TRI_DEV_GROUP_NVALID);
      q.ucount[g] = 0;
    }
    for (int j = t; j < q.member_words; j += UT) member[j] = 0u;
    return;
  }

  // ---- the union of the heads' own picks ----------------------------------
  // The picks are the candidates [P, n - W) in each slice's keep list.
  const int lo = q.n_prompt, hi = n - q.n_recent;
  for (int h = 0; h < q.group && q.bk > 0; ++h) {
    const int32_t* kk = q.keepk + (s0 + h) * static_cast<int64_t>(q.bk);
    for (int j = t; j < q.bk; j += UT) {
      const int v = __ldg(kk + j);
      if (v >= lo && v < hi) atomicOr(&sbits[v >> 5], 1u << (v & 31));
    }
  }
  __syncthreads();
  int cnt = 0;
  for (int j = t; j < q.member_words; j += UT) {
    const uint32_t w = sbits[j];
    member[j] = w;
    cnt += __popc(w);
  }
  const double tot = block_sum(static_cast<double>(cnt), sred);
  if (t == 0) q.ucount[g] = static_cast<int32_t>(tot);
}

// One CTA per slice: mean and population standard deviation of its scores
// over rows [0, n_valid) -- two passes (the mean, then the centred squares),
// fp64 block sums in a fixed order. A thread reads 16 bytes at a time when
// the row is 16-byte aligned and keeps four fp32 partial sums (one per lane
// of the load, each over at most n / 1024 + 1 scores), so its share of at
// most n / 256 scores is summed in shorter chains than one running sum.
__global__ void __launch_bounds__(UT) slice_stats_kernel(const float* __restrict__ scores,
                                                         const int32_t* __restrict__ n_valid, float* stats,
                                                         int n_cap) {
  __shared__ double sred[UW];
  const int t = threadIdx.x;
  const int64_t s = blockIdx.x;
  const int n = min(max(n_valid[s], 0), n_cap);
  const float* row = scores + s * static_cast<int64_t>(n_cap);
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  const int n4 = vec ? (n >> 2) : 0;  // whole 16-byte units; the rest one by one
  const float4* row4 = reinterpret_cast<const float4*>(row);
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 4
  for (int i = t; i < n4; i += UT) {
    const float4 x = __ldcg(row4 + i);
    a0 += x.x;
    a1 += x.y;
    a2 += x.z;
    a3 += x.w;
  }
  for (int i = 4 * n4 + t; i < n; i += UT) a0 += __ldcg(row + i);
  const double mean = (n > 0) ? block_sum((a0 + a1) + (a2 + a3), sred) / n : 0.0;
  const float mf = static_cast<float>(mean);
  float b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
#pragma unroll 4
  for (int i = t; i < n4; i += UT) {
    const float4 x = __ldcg(row4 + i);
    const float d0 = x.x - mf, d1 = x.y - mf, d2 = x.z - mf, d3 = x.w - mf;
    b0 = fmaf(d0, d0, b0);
    b1 = fmaf(d1, d1, b1);
    b2 = fmaf(d2, d2, b2);
    b3 = fmaf(d3, d3, b3);
  }
  for (int i = 4 * n4 + t; i < n; i += UT) {
    const float d = __ldcg(row + i) - mf;
    b0 = fmaf(d, d, b0);
  }
  const float b = (b0 + b1) + (b2 + b3);
  // the centred sum uses the fp32 mean; correct it to the fp64 one
  const double dm = mean - static_cast<double>(mf);
  const double ss = block_sum(b, sred);
  const double var = (n > 0) ? fmax(ss / n - dm * dm, 0.0) : 0.0;
  if (t == 0) {
    stats[s * 2] = mf;
    stats[s * 2 + 1] = static_cast<float>(sqrt(var));
  }
}

}  // namespace

cudaError_t launch_slice_stats(const float* scores, const int32_t* n_valid, float* stats, int n_slices, int n_cap,
                               cudaStream_t st) {
  slice_stats_kernel<<<static_cast<unsigned>(n_slices), UT, 0, st>>>(scores, n_valid, stats, n_cap);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_union_prep(const UnionPrepParams& q, int n_groups, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(q.member_words) * sizeof(uint32_t);
  const cudaError_t e = cudaFuncSetAttribute(union_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  union_prep_kernel<<<static_cast<unsigned>(n_groups), UT, smem, st>>>(q);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tri
