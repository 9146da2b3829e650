// score_heads.cu -- per-query-head TriAttention scores for GQA and the
// statistics of their z-scores.
//
// TriAttention paper summary, section 3.4, "Handling Grouped-Query Attention
// (GQA)": each of the G query heads that share a KV head has its own centre
// statistics, hence its own score of every cached key,
//   S~(g)(i) = Re sum_f W(g)_f e^{i w_f (p_cur - p_i)} conj(k_f) + sum_f n(g)_f |k_f|
// with W(g)_f = c(g)_f G_f and n(g)_f = (1 - R(g)_f) E|q(g)_f| as in the pooled
// score. The scores of head g are z-normalised with their mean and standard
// deviation over all cached keys, and a key's final score is the maximum over
// the G heads (select.cu ranks by it; zmax_scores_kernel writes it out).
//
// This file serves fp32 keys (bf16 keys take the tensor-core kernel of
// score_heads_tc.cu). score_heads_kernel reads every valid row of K once per
// pass and scores up to four heads per pass (the host launches ceil(G/4)
// passes). Per band it
// forms z = e^{i w (p_cur - p)} conj(k) and |k| once; a head then costs two
// paired FMAs for the trigonometric term (Re(W z) = Re W Re z - Im W Im z)
// and one for the norm term, so the arithmetic per key grows with the heads
// while the bytes do not. The tile ring, lane layout and rotation recurrence
// are the pooled kernel's (score.cu).
//
// Statistics: each lane that owns a (key, head) sum also accumulates that
// head's sum and sum of squares, shifted by the first value it saw so that
// fp32 only sees deviations; the CTA combines the lanes in fp64 by a tree of
// fixed shape into one partial per (CTA, head), and heads_stats_kernel adds the
// partials of a slice in order. The results do not depend on scheduling.
#include <cuda_runtime.h>

#include <math.h>

#include "score_common.cuh"
#include "tri_internal.cuh"

namespace tri {
namespace {

constexpr size_t HEADS_BAD_OFF = SCORE_SMEM;  // the paged check's first bad block (16-byte slot)
constexpr size_t HEADS_JUMP_OFF = HEADS_BAD_OFF + 16;
constexpr size_t HEADS_SMEM = HEADS_JUMP_OFF + MAX_BANDS / 2 * sizeof(float4);

// Sums a[0..NU) over the TPK lanes of a key group. Each lane ends with RPL =
// max(1, NU / TPK) consecutive sums, entries idx .. idx + RPL - 1; when NU <
// TPK, lanes that differ only in their low TPK/NU bits hold the same entry.
template <int TPK, int NU>
__device__ __forceinline__ void reduce_heads(float (&a)[NU], int lane, int& idx,
                                             float (&out)[(NU >= TPK) ? NU / TPK : 1]) {
  constexpr int RPL = (NU >= TPK) ? NU / TPK : 1;
  idx = 0;
  int m = TPK / 2;
#pragma unroll
  for (int v = NU; v > RPL; v >>= 1) {
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
#pragma unroll
  for (int r = 0; r < RPL; ++r) out[r] = a[r];
  if (NU < TPK) {
#pragma unroll
    for (int mm = TPK / NU / 2; mm >= 1; mm >>= 1) out[0] += __shfl_xor_sync(FULL_MASK, out[0], mm);
  }
}

template <typename T, int D, int STYLE, int PM, int GH>
__global__ void __launch_bounds__(SCORE_THREADS, 2)
    score_heads_kernel(const __grid_constant__ ScoreParams p) {
  using G = Geo<T, D>;
  constexpr bool EXPLICIT_POS = PM == POS_EXPLICIT, POST = PM == POS_POST_ROPE;
  constexpr int F = G::F, BPT = G::BPT, NP = BPT / 2, TPK = G::TPK, KPW = G::KPW;
  constexpr int ROW_BYTES = G::ROW_BYTES, TILE_ROWS = G::TILE_ROWS, RPW = G::RPW, STEPS = G::STEPS;
  constexpr int GHP = (GH == 3) ? 4 : GH;  // heads padded to a power of two for the reduction
  constexpr int HS = 2;                    // keys per lane between reductions
  constexpr int NU = GHP * HS;
  constexpr int RPL = (NU >= TPK) ? NU / TPK : 1;
  static_assert(STEPS % HS == 0, "steps per reduction");
  static_assert(GH * 3 * SCORE_THREADS * sizeof(double) <= RING_BYTES, "statistics rows fit in the ring");
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  RingCtrl& rc = *reinterpret_cast<RingCtrl*>(smem + RING_BYTES);
  int* sbad = reinterpret_cast<int*>(smem + HEADS_BAD_OFF);
  // per band pair: the tile-to-tile rotation (re0, re1, im0, im1)
  float4* sjump = reinterpret_cast<float4*>(smem + HEADS_JUMP_OFF);

  const int64_t s = blockIdx.x / p.tiles_per_slice;
  const int ct = blockIdx.x % p.tiles_per_slice;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  double* my_part = p.partials + ((s * p.tiles_per_slice + ct) * p.group + p.head0) * 3;

  const int n = p.n_valid[s];
  const bool bad = n > p.n_cap || n < 0;
  if (bad && threadIdx.x == 0 && ct == 0) set_status(p.dev_status, TRI_DEV_NVALID_OVER_CAP);
  const int c0 = ct * p.rows_per_cta;
  const int c1 = bad ? c0 : min((ct + 1) * p.rows_per_cta, n);
  if (c0 >= c1) {  // nothing to score: an empty partial (uniform over the CTA)
    if (threadIdx.x < 3 * GH) my_part[threadIdx.x] = 0.0;
    return;
  }
  const int ntiles = (c1 - c0 + TILE_ROWS - 1) / TILE_ROWS;
  const unsigned char* kbase = static_cast<const unsigned char*>(p.k);
  const int64_t sbase = p.rows.slice_base(s);
  const int32_t* trow = p.rows.seq_table(s);
  if (!p.rows.blocks_ok(trow, c0, c1, sbad)) {  // uniform over the CTA
    if (threadIdx.x == 0) set_status(p.dev_status, TRI_DEV_BAD_BLOCK);
    if (threadIdx.x < 3 * GH) my_part[threadIdx.x] = 0.0;
    return;
  }

  // one bulk copy per run of rows contiguous in memory (see score.cu)
  auto issue = [&](int u) {
    const int r0 = c0 + u * TILE_ROWS;
    const int rows = min(TILE_ROWS, c1 - r0);
    uint64_t* bar = &rc.full[u % STAGES];
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(rows * ROW_BYTES));
    unsigned char* dst = ring + (u % STAGES) * TILE_BYTES;
    for (int done = 0; done < rows;) {
      const int run = p.rows.run(r0 + done, rows - done);
      bulk_g2s(dst + done * ROW_BYTES, kbase + p.rows.row(sbase, trow, r0 + done), static_cast<uint32_t>(run * ROW_BYTES),
               bar);
      done += run;
    }
  };
  if (threadIdx.x == 0) ring_init(rc, ntiles);
  if (threadIdx.x < F / 2) {
    const int f = 2 * threadIdx.x;
    sjump[threadIdx.x] = make_float4(p.jump_re[f], p.jump_re[f + 1], p.jump_im[f], p.jump_im[f + 1]);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int u = 0; u < min(STAGES, ntiles); ++u) issue(u);
  }

  // ---- per-lane constants: bands c*BPT .. c*BPT+BPT-1 as NP pairs ----------
  const int c = lane % TPK;
  const int kq = lane / TPK;
  const int lh = static_cast<int>(s % p.lh_count);
  const int64_t seq = s / p.lh_count;
  const int64_t pc = p.p_cur[seq];
  float2 WR[GH][NP], WI[GH][NP], NW[GH][NP];
  float2 ER[NP], EI[NP], SR[NP], SI[NP], NSI[NP];
  uint64_t nu[BPT];
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    float er[2] = {0.f, 0.f}, ei[2] = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int f = c * BPT + 2 * q + h;
      nu[2 * q + h] = p.nu[f];
      if (!EXPLICIT_POS) {
        // post-RoPE: the constant e^{i w p_cur}; slot positions: the first key's rotation
        const int64_t delta = POST ? pc : pc - (c0 + warp * RPW + kq);
        const float2 e = turns_rotation_accurate(delta, p.nu[f]);
        er[h] = e.x;
        ei[h] = e.y;
      }
    }
#pragma unroll
    for (int g = 0; g < GH; ++g) {
      float wr[2], wi[2], nw[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int f = c * BPT + 2 * q + h;
        const int64_t row = (static_cast<int64_t>(lh) * p.group + p.head0 + g) * F + f;
        const float2 cf = reinterpret_cast<const float2*>(p.center)[row];
        const float m = p.mean_norm[row];
        const float R = p.mrl[row];
        nw[h] = (p.norm_mode == TRI_NORM_UNWEIGHTED) ? m : (1.0f - R) * m;
        float2 w = cmul(cf, make_float2(p.g_re[f], p.g_im[f]));
        if (POST) w = cmul(w, make_float2(er[h], ei[h]));  // fold the constant rotation in
        wr[h] = w.x;
        wi[h] = w.y;
      }
      WR[g][q] = f2(wr[0], wr[1]);
      WI[g][q] = f2(wi[0], wi[1]);
      NW[g][q] = f2(nw[0], nw[1]);
    }
    const int f0 = c * BPT + 2 * q;
    ER[q] = f2(er[0], er[1]);
    EI[q] = f2(ei[0], ei[1]);
    SR[q] = f2(p.step_re[f0], p.step_re[f0 + 1]);
    SI[q] = f2(p.step_im[f0], p.step_im[f0 + 1]);
    NSI[q] = f2(-p.step_im[f0], -p.step_im[f0 + 1]);
  }

  float* out = p.scores_g + (s * p.group + p.head0) * static_cast<int64_t>(p.n_cap);
  const int32_t* pos = EXPLICIT_POS ? p.pos + s * static_cast<int64_t>(p.n_cap) : nullptr;
  // lanes that own their reduced sums (the others hold copies)
  const bool own = (NU >= TPK) || (c % (TPK / NU)) == 0;
  float sh = 0.f, s1 = 0.f, s2 = 0.f;  // this lane's head: shift, shifted sum and sum of squares
  int cnt = 0;
  int lane_head = -1;

  for (int t = 0; t < ntiles; ++t) {
    const int st = t % STAGES;
    if (!ring_wait(rc, t, lane)) break;
    {
      const unsigned char* tile = ring + st * TILE_BYTES;
      const int rbase = warp * RPW + kq;
      int pp[STEPS];
      if (EXPLICIT_POS) {
#pragma unroll
        for (int j = 0; j < STEPS; ++j) {
          const int r = c0 + t * TILE_ROWS + rbase + j * KPW;
          pp[j] = (r < c1) ? __ldg(pos + r) : 0;
        }
      }
#pragma unroll
      for (int h0 = 0; h0 < STEPS; h0 += HS) {
      float acc[NU];
#pragma unroll
      for (int e = 0; e < NU; ++e) acc[e] = 0.f;
#pragma unroll
      for (int jj = 0; jj < HS; ++jj) {
        const int j = h0 + jj;
        const int rt = rbase + j * KPW;
        const bool valid = c0 + t * TILE_ROWS + rt < c1;
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (valid) raw = lds_chunk<T, D, STYLE>(tile + rt * ROW_BYTES, c);
        float re[BPT], im[BPT];
        decode_chunk<T, STYLE>(raw, re, im);
        float2 a[GH];  // each starts with the first band pair's product (no zeroing)
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          const float2 RE = f2(re[2 * q], re[2 * q + 1]);
          const float2 IM = f2(im[2 * q], im[2 * q + 1]);
          const float2 sq = __ffma2_rn(IM, IM, __fmul2_rn(RE, RE));
          const float2 mag = f2(sqrt_approx(sq.x), sqrt_approx(sq.y));
          if (POST) {
            // Re(W e^{i w p_cur} conj(k~)) = Re(W') Re k~ + Im(W') Im k~
#pragma unroll
            for (int g = 0; g < GH; ++g) {
              a[g] = (q == 0) ? __fmul2_rn(WR[g][q], RE) : __ffma2_rn(WR[g][q], RE, a[g]);
              a[g] = __ffma2_rn(WI[g][q], IM, a[g]);
              a[g] = __ffma2_rn(NW[g][q], mag, a[g]);
            }
            continue;
          }
          float2 er, ei;
          if (EXPLICIT_POS) {
            const float2 r0 = turns_rotation_fast(pc - pp[j], nu[2 * q]);
            const float2 r1 = turns_rotation_fast(pc - pp[j], nu[2 * q + 1]);
            er = f2(r0.x, r1.x);
            ei = f2(r0.y, r1.y);
          } else {
            er = ER[q];
            ei = EI[q];
            ER[q] = __ffma2_rn(er, SR[q], __fmul2_rn(ei, NSI[q]));
            EI[q] = __ffma2_rn(er, SI[q], __fmul2_rn(ei, SR[q]));
          }
          // z = e conj(k): Re z = er kr + ei ki; -Im z = er ki - ei kr
          const float2 zr = __ffma2_rn(er, RE, __fmul2_rn(ei, IM));
          const float2 zn = __ffma2_rn(er, IM, __fmul2_rn(ei, f2(-RE.x, -RE.y)));
#pragma unroll
          for (int g = 0; g < GH; ++g) {
            a[g] = (q == 0) ? __fmul2_rn(WR[g][q], zr) : __ffma2_rn(WR[g][q], zr, a[g]);
            a[g] = __ffma2_rn(WI[g][q], zn, a[g]);
            a[g] = __ffma2_rn(NW[g][q], mag, a[g]);
          }
        }
#pragma unroll
        for (int g = 0; g < GH; ++g) acc[g * HS + jj] = a[g].x + a[g].y;
      }
      int idx;
      float v[RPL];
      reduce_heads<TPK, NU>(acc, lane, idx, v);
#pragma unroll
      for (int r = 0; r < RPL; ++r) {
        const int e = idx + r;
        const int g = e / HS, j = h0 + e % HS;
        const int row = c0 + t * TILE_ROWS + rbase + j * KPW;
        if (own && g < GH && row < c1) {
          __stcs(out + static_cast<int64_t>(g) * p.n_cap + row, v[r]);
          if (cnt == 0) sh = v[r];
          const float dv = v[r] - sh;
          s1 += dv;
          s2 = fmaf(dv, dv, s2);
          ++cnt;
          lane_head = g;
        }
      }
      }
      if (PM == POS_SLOT) {
        // from this lane's last key of tile t to its first key of tile t + 1
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          const float4 jq = sjump[c * NP + q];
          const float2 jr = f2(jq.x, jq.y), ji = f2(jq.z, jq.w), nji = f2(-jq.z, -jq.w);
          const float2 er = ER[q], ei = EI[q];
          ER[q] = __ffma2_rn(er, jr, __fmul2_rn(ei, nji));
          EI[q] = __ffma2_rn(er, ji, __fmul2_rn(ei, jr));
        }
      }
    }
    ring_release(rc, t, ntiles, lane, issue);
    if (ring_failed(rc)) break;
  }
  __syncthreads();
  ring_drain(rc, p.dev_status);

  // ---- statistics partials of this CTA, per head, in fp64 -------------------
  // Thread u's plain sums go to column u of its head's three rows (zeros in
  // the other heads' rows), and a tree of fixed shape adds each row's
  // columns: no long serial chain on the slow fp64 pipe. The drained ring
  // holds the rows.
  __syncthreads();
  double* sx = reinterpret_cast<double*>(ring);  // [GH][3][SCORE_THREADS]
  {
    const double dn = cnt, dsh = sh, ds1 = s1;
    const double e0 = dn * dsh + ds1;                                        // sum
    const double e1 = dn * dsh * dsh + 2.0 * dsh * ds1 + static_cast<double>(s2);  // sum of squares
#pragma unroll
    for (int g = 0; g < GH; ++g) {
      const bool mine = g == lane_head;
      sx[(g * 3 + 0) * SCORE_THREADS + threadIdx.x] = mine ? e0 : 0.0;
      sx[(g * 3 + 1) * SCORE_THREADS + threadIdx.x] = mine ? e1 : 0.0;
      sx[(g * 3 + 2) * SCORE_THREADS + threadIdx.x] = mine ? dn : 0.0;
    }
  }
  __syncthreads();
  for (int stride = SCORE_THREADS / 2; stride >= 1; stride >>= 1) {
    for (int i = threadIdx.x; i < GH * 3 * stride; i += SCORE_THREADS) {
      const int r = i / stride, k = i % stride;
      sx[r * SCORE_THREADS + k] += sx[r * SCORE_THREADS + k + stride];
    }
    __syncthreads();
  }
  if (threadIdx.x < 3 * GH) my_part[threadIdx.x] = sx[threadIdx.x * SCORE_THREADS];
}

// One thread per (slice, head): the partials of the slice's CTAs in order.
__global__ void heads_stats_kernel(const double* __restrict__ partials, float* __restrict__ stats, int n_slices,
                                   int tiles_per_slice, int group) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(n_slices) * group) return;
  const int64_t s = i / group;
  const int g = static_cast<int>(i % group);
  double a = 0.0, b = 0.0, n = 0.0;
  for (int ct = 0; ct < tiles_per_slice; ++ct) {
    const double* q = partials + ((s * tiles_per_slice + ct) * group + g) * 3;
    a += q[0];
    b += q[1];
    n += q[2];
  }
  float mu = 0.f, sd = 0.f;
  if (n > 0.0) {
    const double m = a / n;
    const double var = fmax(b / n - m * m, 0.0);  // population variance
    mu = static_cast<float>(m);
    sd = static_cast<float>(sqrt(var));
  }
  stats[2 * i] = mu;
  stats[2 * i + 1] = sd;
}

// The final score max_g z_g of every valid row (for callers that want the
// values; the selection computes them on the fly in the same way).
__global__ void zmax_scores_kernel(const float* __restrict__ scores_g, const float* __restrict__ stats,
                                   const int32_t* __restrict__ n_valid, int nv_stride, float* __restrict__ out,
                                   int n_cap, int group, int blocks_per_slice) {
  const int64_t s = blockIdx.x / blocks_per_slice;
  const int i = (blockIdx.x % blocks_per_slice) * blockDim.x + threadIdx.x;
  const int n = min(n_valid[s * nv_stride], n_cap);
  if (i >= n) return;
  float best = 0.f;
  for (int g = 0; g < group; ++g) {
    const float mu = stats[(s * group + g) * 2];
    const float inv = head_inv_std(stats[(s * group + g) * 2 + 1]);
    const float z = head_z(__ldg(scores_g + (s * group + g) * static_cast<int64_t>(n_cap) + i), mu, inv);
    best = (g == 0) ? z : fmaxf(best, z);
  }
  out[s * static_cast<int64_t>(n_cap) + i] = best;
}

template <typename T, int D, int STYLE, int PM, int GH>
cudaError_t launch_one(const ScoreParams& p, int n_slices, cudaStream_t st) {
  auto kern = score_heads_kernel<T, D, STYLE, PM, GH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(HEADS_SMEM));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(n_slices) * p.tiles_per_slice));
  kern<<<grid, SCORE_THREADS, HEADS_SMEM, st>>>(p);
  note_launch();
  return cudaGetLastError();
}

template <typename T, int D, int STYLE, int PM>
cudaError_t launch_heads(const ScoreParams& p, int n_heads, int n_slices, cudaStream_t st) {
  switch (n_heads) {
    case 1: return launch_one<T, D, STYLE, PM, 1>(p, n_slices, st);
    case 2: return launch_one<T, D, STYLE, PM, 2>(p, n_slices, st);
    case 3: return launch_one<T, D, STYLE, PM, 3>(p, n_slices, st);
    case 4: return launch_one<T, D, STYLE, PM, 4>(p, n_slices, st);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, int D, int STYLE>
cudaError_t launch_pm(const ScoreParams& p, int n_heads, int pm, int n_slices, cudaStream_t st) {
  if (pm == POS_POST_ROPE) return launch_heads<T, D, STYLE, POS_POST_ROPE>(p, n_heads, n_slices, st);
  if (pm == POS_EXPLICIT) return launch_heads<T, D, STYLE, POS_EXPLICIT>(p, n_heads, n_slices, st);
  return launch_heads<T, D, STYLE, POS_SLOT>(p, n_heads, n_slices, st);
}

template <typename T, int D>
cudaError_t launch_style(const ScoreParams& p, int n_heads, tri_rope_style style, int pm, int n_slices,
                         cudaStream_t st) {
  if (style == TRI_ROPE_INTERLEAVED) return launch_pm<T, D, TRI_ROPE_INTERLEAVED>(p, n_heads, pm, n_slices, st);
  return launch_pm<T, D, TRI_ROPE_HALF>(p, n_heads, pm, n_slices, st);
}

}  // namespace

cudaError_t launch_score_heads(const ScoreParams& p, int n_heads, tri_dtype dt, int head_dim,
                               tri_rope_style style, int pos_mode, int n_slices, cudaStream_t st) {
  if (dt != TRI_F32) return cudaErrorInvalidValue;  // bf16 keys: score_heads_tc.cu
  if (head_dim == 128) return launch_style<float, 128>(p, n_heads, style, pos_mode, n_slices, st);
  return launch_style<float, 64>(p, n_heads, style, pos_mode, n_slices, st);
}

cudaError_t launch_heads_stats(const double* partials, float* stats, int n_slices, int tiles_per_slice,
                               int group, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(n_slices) * group;
  const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
  heads_stats_kernel<<<blocks, 256, 0, st>>>(partials, stats, n_slices, tiles_per_slice, group);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_zmax_scores(const float* scores_g, const float* stats, const int32_t* n_valid, int nv_stride,
                               float* out, int n_blocks, int n_cap, int group, cudaStream_t st) {
  const int bps = (n_cap + 255) / 256;
  const int64_t blocks = static_cast<int64_t>(bps) * n_blocks;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  zmax_scores_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(scores_g, stats, n_valid, nv_stride, out,
                                                                     n_cap, group, bps);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tri
