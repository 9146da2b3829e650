// score_core.cuh -- one CTA of the TriAttention score (score.cu launches it
// as the score kernel; compress.cu runs it before the slice's selection).
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
//   * one CTA streams a contiguous run of a slice's rows through a 2-stage
//     ring of 32 KB shared-memory tiles, each filled by one bulk async copy
//     (TMA, non-tensor) that completes on an mbarrier; thread 0 refills a
//     stage as soon as the CTA has consumed it (64 KB per CTA, 192 KB per
//     SM; 32 KB tiles amortise each tile's waits, barrier and reduction over
//     twice the keys of 16 KB ones);
//   * a key row is split across TPK lanes, each lane owning BPT consecutive
//     bands (one 16-byte shared load per key); band constants live in
//     registers as fp32 pairs so that two bands share one paired
//     (f32x2) multiply-add;
//   * for implicit positions the rotation e^{i w_f (p_cur - p)} is advanced
//     by one complex multiply per key (anchored once per CTA from an exact
//     64-bit fixed-point phase); with explicit positions it is evaluated per
//     key from the fixed-point phase;
//   * each warp handles RPW rows of a tile as STEPS keys per lane; the STEPS
//     partial sums are reduced across the TPK lanes with a transposed
//     butterfly that leaves consecutive scores in consecutive lanes.
// Every wait on a tile is bounded in wall-clock time; a timeout records
// TRI_DEV_TIMEOUT, drains the copies in flight and leaves the rest unscored.

#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "score_common.cuh"
#include "tri_internal.cuh"

namespace tri {
namespace {

// Reduce-scatter of a[0..NU) over the TPK lanes of one key group. On return,
// every lane holds the full sum of entry `idx` (lanes that differ only in the
// bits below TPK/NU hold the same entry).
template <int TPK, int NU>
__device__ __forceinline__ float reduce_scatter(float (&a)[NU], int lane, int& idx) {
  idx = 0;
  int m = TPK / 2;
#pragma unroll
  for (int v = NU; v > 1; v >>= 1) {
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
  for (int mm = TPK / NU / 2; mm >= 1; mm >>= 1) r += __shfl_xor_sync(FULL_MASK, r, mm);
  return r;
}

// One score CTA: run `ct` of slice s (rows [ct rows_per_cta, (ct + 1)
// rows_per_cta) clipped to the candidates [P, n - W)), by all SCORE_THREADS
// threads, with SCORE_SMEM bytes of dynamic shared memory at `smem`. Every
// early return is uniform over the CTA. STREAM_OUT stores the scores with an
// evict-first hint (nothing in the same kernel reads them back).
template <typename T, int D, int STYLE, int PM, bool PAGED, bool STREAM_OUT>
__device__ __forceinline__ void score_cta(const ScoreParams& p, unsigned char* smem, int64_t s, int ct) {
  using G = Geo<T, D>;
  constexpr bool EXPLICIT_POS = PM == POS_EXPLICIT, POST = PM == POS_POST_ROPE;
  constexpr int F = G::F, BPT = G::BPT, NP = BPT / 2, TPK = G::TPK, KPW = G::KPW;
  constexpr int ROW_BYTES = G::ROW_BYTES, TILE_ROWS = G::TILE_ROWS, RPW = G::RPW, STEPS = G::STEPS;
  unsigned char* ring = smem;
  RingCtrl& rc = *reinterpret_cast<RingCtrl*>(smem + RING_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n = p.n_valid[s];
  if (n > p.n_cap || n < 0) {
    if (threadIdx.x == 0 && ct == 0) set_status(p.dev_status, TRI_DEV_NVALID_OVER_CAP);
    return;
  }
  const int c0 = max(ct * p.rows_per_cta, p.n_prompt);
  const int c1 = min((ct + 1) * p.rows_per_cta, n - p.n_recent);
  if (c0 >= c1) return;  // uniform over the CTA
  const int ntiles = (c1 - c0 + TILE_ROWS - 1) / TILE_ROWS;
  const unsigned char* kbase = static_cast<const unsigned char*>(p.k);
  const int64_t sbase = p.rows.slice_base(s);
  const int32_t* trow = p.rows.seq_table(s);
  // paged: the CTA's table entries, checked and cached in shared memory
  constexpr int TAB = 32 * 128 / 16 + 2;  // entries for the most rows a CTA takes, 16-row blocks
  __shared__ int32_t stab[PAGED ? TAB : 1];
  const int b0 = PAGED ? (c0 >> p.rows.block_shift) : 0;
  if (PAGED) {
    __shared__ int bad_block;
    if (!p.rows.blocks_ok(trow, c0, c1, &bad_block, stab)) {  // uniform over the CTA
      if (threadIdx.x == 0) set_status(p.dev_status, TRI_DEV_BAD_BLOCK);
      return;
    }
  }
  const unsigned char* src = kbase + sbase + static_cast<int64_t>(c0) * ROW_BYTES;  // contiguous slices

  // Tile u = rows [c0 + u TILE_ROWS, ...): one bulk copy by thread 0
  // (contiguous slices), or one per run of rows inside a block, issued by the
  // lanes of warp 0 together (paged).
  auto issue = [&](int u) {
    const int r0 = c0 + u * TILE_ROWS;
    const int rows = min(TILE_ROWS, c1 - r0);
    uint64_t* bar = &rc.full[u % STAGES];
    if (!PAGED || lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(rows * ROW_BYTES));
    if (PAGED) __syncwarp();
    unsigned char* dst = ring + (u % STAGES) * TILE_BYTES;
    if (!PAGED) {
      bulk_g2s(dst, src + static_cast<int64_t>(u) * TILE_BYTES, static_cast<uint32_t>(rows * ROW_BYTES), bar);
      return;
    }
    // paged: called by all of warp 0; lane i copies the tile's i-th block
    // piece (the first starts inside a block, the others at row 0), so the
    // pieces go out together instead of one after another
    const int bs = p.rows.block_size, sh = p.rows.block_shift;
    const int o0 = r0 & (bs - 1);
    const int nruns = (o0 + rows + bs - 1) >> sh;  // at most TILE_ROWS / 16 + 1
    if (lane < nruns) {
      const int start = (lane == 0) ? 0 : lane * bs - o0;  // first row of the piece in the tile
      const int o = (lane == 0) ? o0 : 0;
      const int run = min(bs - o, rows - start);
      bulk_g2s(dst + start * ROW_BYTES,
               kbase + sbase + static_cast<int64_t>(stab[(r0 >> sh) - b0 + lane]) * p.rows.block_bytes + o * ROW_BYTES,
               static_cast<uint32_t>(run * ROW_BYTES), bar);
    }
  };
  if (threadIdx.x == 0) ring_init(rc, ntiles);
  __syncthreads();
  if (PAGED ? warp == 0 : threadIdx.x == 0) {
    for (int u = 0; u < min(STAGES, ntiles); ++u) issue(u);
  }

  // ---- per-lane band constants (bands c*BPT .. c*BPT+BPT-1, as NP pairs) --
  const int c = lane % TPK;   // band group of this lane
  const int kq = lane / TPK;  // key of the warp step this lane works on
  const int lh = static_cast<int>(s % p.lh_count);
  const int64_t seq = s / p.lh_count;
  const int64_t pc = p.p_cur[seq];
  float2 WR[NP], WI[NP], DR[NP], DI[NP], SR[NP], SI[NP], NSI[NP], JR[NP], JI[NP], NW[NP];
  uint64_t nu[BPT];
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    float wr[2], wi[2], nw[2], dr[2], di[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int f = c * BPT + 2 * q + h;
      const float2 cf = reinterpret_cast<const float2*>(p.center)[static_cast<int64_t>(lh) * F + f];
      const float m = p.mean_norm[static_cast<int64_t>(lh) * F + f];
      const float R = p.mrl[static_cast<int64_t>(lh) * F + f];
      nw[h] = (p.norm_mode == TRI_NORM_UNWEIGHTED) ? m : (1.0f - R) * m;
      const float2 w = cmul(cf, make_float2(p.g_re[f], p.g_im[f]));
      wr[h] = w.x;
      wi[h] = w.y;
      nu[2 * q + h] = p.nu[f];
      if (!EXPLICIT_POS) {
        // post-RoPE: the constant e^{i w p_cur}; slot positions: the first key's rotation
        const int64_t delta = POST ? pc : pc - (c0 + warp * RPW + kq);
        const float2 d = cmul(w, turns_rotation_accurate(delta, p.nu[f]));
        dr[h] = d.x;
        di[h] = d.y;
      }
    }
    WR[q] = f2(wr[0], wr[1]);
    WI[q] = f2(wi[0], wi[1]);
    NW[q] = f2(nw[0], nw[1]);
    const int f0 = c * BPT + 2 * q;
    SR[q] = f2(p.step_re[f0], p.step_re[f0 + 1]);
    SI[q] = f2(p.step_im[f0], p.step_im[f0 + 1]);
    NSI[q] = f2(-p.step_im[f0], -p.step_im[f0 + 1]);
    JR[q] = f2(p.jump_re[f0], p.jump_re[f0 + 1]);
    JI[q] = f2(p.jump_im[f0], p.jump_im[f0 + 1]);
    if (!EXPLICIT_POS) {
      DR[q] = f2(dr[0], dr[1]);
      DI[q] = f2(di[0], di[1]);
    } else {
      DR[q] = DI[q] = f2(0.f, 0.f);
    }
  }

  float* out = p.scores + s * static_cast<int64_t>(p.n_cap);
  const int32_t* pos = EXPLICIT_POS ? p.pos + s * static_cast<int64_t>(p.n_cap) : nullptr;

  // One tile's keys of this lane. FULL: every row of the tile lies in the
  // run (all tiles but possibly the last), so no key needs a range check.
  // Only contiguous caches with slot or post-RoPE positions take a separate
  // full-tile body: for paged caches and explicit positions the second copy
  // of the larger body measured slower.
  auto score_tile = [&](const int t, auto full_tag) {
    constexpr bool FULL = decltype(full_tag)::value;
    {
      const unsigned char* tile = ring + (t % STAGES) * TILE_BYTES;
      const int rbase = warp * RPW + kq;  // row within the tile of this lane's first key
      int pp[STEPS];
      if (EXPLICIT_POS) {
#pragma unroll
        for (int j = 0; j < STEPS; ++j) {
          const int r = c0 + t * TILE_ROWS + rbase + j * KPW;
          pp[j] = (FULL || r < c1) ? __ldg(pos + r) : 0;
        }
      }
      float acc[STEPS];
#pragma unroll
      for (int j = 0; j < STEPS; ++j) {
        const int rt = rbase + j * KPW;
        uint4 raw;
        if (FULL) {
          raw = lds_chunk<T, D, STYLE>(tile + rt * ROW_BYTES, c);
        } else {
          raw = make_uint4(0u, 0u, 0u, 0u);
          if (c0 + t * TILE_ROWS + rt < c1) raw = lds_chunk<T, D, STYLE>(tile + rt * ROW_BYTES, c);
        }
        float re[BPT], im[BPT];
        decode_chunk<T, STYLE>(raw, re, im);
        float2 a2;  // starts with the first band pair's product (no zeroing)
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          const float2 RE = f2(re[2 * q], re[2 * q + 1]);
          const float2 IM = f2(im[2 * q], im[2 * q + 1]);
          float2 dr, di;
          if (EXPLICIT_POS) {
            const float2 r0 = turns_rotation_fast(pc - pp[j], nu[2 * q]);
            const float2 r1 = turns_rotation_fast(pc - pp[j], nu[2 * q + 1]);
            const float2 C = f2(r0.x, r1.x), S = f2(r0.y, r1.y);
            dr = __ffma2_rn(WR[q], C, __fmul2_rn(WI[q], f2(-S.x, -S.y)));
            di = __ffma2_rn(WR[q], S, __fmul2_rn(WI[q], C));
          } else if (POST) {
            dr = DR[q];
            di = DI[q];
          } else {
            dr = DR[q];
            di = DI[q];
            DR[q] = __ffma2_rn(dr, SR[q], __fmul2_rn(di, NSI[q]));
            DI[q] = __ffma2_rn(dr, SI[q], __fmul2_rn(di, SR[q]));
          }
          a2 = (q == 0) ? __fmul2_rn(dr, RE) : __ffma2_rn(dr, RE, a2);
          a2 = __ffma2_rn(di, IM, a2);
          const float2 sq = __ffma2_rn(IM, IM, __fmul2_rn(RE, RE));
          a2 = __ffma2_rn(NW[q], f2(sqrt_approx(sq.x), sqrt_approx(sq.y)), a2);
        }
        acc[j] = a2.x + a2.y;
      }
      if (PM == POS_SLOT) {
        // from this lane's last key of tile t to its first key of tile t + 1
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          const float2 dr = DR[q], di = DI[q];
          const float2 nji = f2(-JI[q].x, -JI[q].y);
          DR[q] = __ffma2_rn(dr, JR[q], __fmul2_rn(di, nji));
          DI[q] = __ffma2_rn(dr, JI[q], __fmul2_rn(di, JR[q]));
        }
      }
      int idx;
      const float v = reduce_scatter<TPK, STEPS>(acc, lane, idx);
      const int r = c0 + t * TILE_ROWS + rbase + idx * KPW;
      if ((c % (TPK / STEPS)) == 0 && (FULL || r < c1)) {
        if (STREAM_OUT) __stcs(out + r, v); else out[r] = v;
      }
    }
  };

  for (int t = 0; t < ntiles; ++t) {
    // a warp whose wait timed out still reaches the barrier below
    if (ring_wait(rc, t, lane)) {
      if constexpr (!PAGED && !EXPLICIT_POS) {
        if (c0 + (t + 1) * TILE_ROWS <= c1) score_tile(t, std::true_type{});
        else score_tile(t, std::false_type{});
      } else {
        score_tile(t, std::false_type{});
      }
    }
    // The kernel is near its issue limit and keeps its warps in step: the
    // whole CTA finishes a stage before thread 0 refills it (measured a little
    // faster here, contiguous or paged, than the per-warp release the heads
    // kernel uses).
    __syncthreads();
    if (ring_failed(rc)) break;
    if ((PAGED ? warp == 0 : threadIdx.x == 0) && t + STAGES < ntiles) {
      fence_proxy_async_smem();
      issue(t + STAGES);
      if (threadIdx.x == 0) rc.issued = t + STAGES + 1;
    }
  }
  __syncthreads();
  ring_drain(rc, p.dev_status);
}

}  // namespace
}  // namespace tri
