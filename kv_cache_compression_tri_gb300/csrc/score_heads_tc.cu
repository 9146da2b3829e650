// score_heads_tc.cu -- per-query-head TriAttention scores for GQA, bf16 keys,
// with the contraction over the heads on the tensor cores.
//
// TriAttention paper summary, section 3.4, "Handling Grouped-Query Attention
// (GQA)": every query head g of a group scores every cached key,
//   S~(g)(i) = Re sum_f W(g)_f e^{i w_f (p_cur - p_i)} conj(k_f) + sum_f n(g)_f |k_f|,
// W(g)_f = c(g)_f G_f, n(g)_f = (1 - R(g)_f) E|q(g)_f| (the pooled score's
// coefficients, per query head). With z_f = e^{i w_f (p_cur - p_i)} conj(k_f),
//   S~(g)(i) = sum_f Re W(g)_f Re z_f + Im W(g)_f (-Im z_f) + n(g)_f |k_f|,
// i.e. the dot product of a key's 3F features x = (Re z, -Im z, |k|) with the
// head's coefficient column. The CUDA cores read each key once and form x
// (one rotation per band and key, as in the pooled kernel); for a block of
// 128 keys the [128 x 3F] feature matrix times the [3F x 16] coefficient
// matrix (up to eight heads) is one chain of tcgen05.mma (kind::f16, fp32
// accumulation in tensor memory), so the per-key cost no longer grows with
// the number of heads. Post-RoPE keys: x = (Re k~, Im k~, |k~|) and the
// constant e^{i w_f p_cur} is folded into the coefficients.
//
// Precision. Features are rounded once to fp16 (relative 2^-11). Each
// coefficient is scaled by a power of two per head (its largest coefficient
// lands in [2^13, 2^14)) and split into an fp16 pair hi + lo, which fill
// columns 2g and 2g+1; the sum of the two accumulators carries the
// coefficients to about 2^-22. The score's error is then at most about
// 2^-11 * sqrt(2) * sum_f E|q(g)_f| |k_f| plus fp32 accumulation. A band with
// |k_f| >= 65520 does not fit fp16: its score comes out non-finite and the
// z-score selection reports TRI_DEV_NAN_SCORE.
//
// CTA: one per SM, a run of up to 16384 rows of one slice, with two groups
// of four feature warps, an MMA warp and a copy warp (ten warps: at most
// three share a scheduler, so a thread may hold up to 168 registers and each
// feature warp forms 32 keys of a block with the loads of all of them in
// flight). The copy warp streams
// key tiles of 128 rows into a 64 KB ring (bulk async copies completing on
// "full" mbarriers; a stage is refilled once its "empty" mbarrier says the
// tile was taken). Each tile is one MMA block; the two groups take
// alternate tiles. A group first loads its lanes' chunks of the tile into
// registers and hands the stage back, so the ring's bytes stay in flight
// rather than waiting for arithmetic. Blocks rotate through three operand
// buffers and three accumulators (block t uses buffer t % 3): the group
// forms the features of block t in the operands' 128-byte-swizzled K-major
// layout once block t - 3 (the other group's) is done with that buffer, and
// arrives on "A full"; the MMA warp issues the block's MMAs into accumulator
// t % 3 and commits them to "MMA done"; the group then reads out its
// previous block t - 2, whose MMAs ran while it formed block t -- each warp
// 32 keys (its quarter of the tensor-memory lanes) and every head --
// stores the scores, adds them to the heads' statistics (sum and sum of
// squares shifted by the thread's first value, folded in fp64 by a tree of
// fixed shape into one partial per CTA and head) and
// arrives on "D free", which the MMA warp waits for before block t + 1
// overwrites that accumulator. No group waits for its own block's MMAs, no
// CTA barrier in the loop; every wait is bounded.
//
// Phase order. A parity wait cannot tell a phase from the one two later, so
// every waiter observes every phase of the mbarriers it waits on, in order:
// the ring holds one group's tiles per stage (tile t in stage t % NST, NST
// even), so each stage's "full" and "empty" phases are one group's and one
// copy thread's; each group waits for every block's "MMA done" in block
// order (block t - 3, the other group's, before forming block t; its own
// block t - 2 for the read-out); the MMA warp takes every "A full" and
// "D free" phase in order.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <math.h>

#include "score_common.cuh"
#include "tri_internal.cuh"
#include "umma.cuh"

namespace tri {
namespace {

constexpr int TC_GROUP_WARPS = 4;                        // feature warps per group
constexpr int TC_GROUP_THREADS = TC_GROUP_WARPS * 32;
constexpr int TC_FEAT_WARPS = 2 * TC_GROUP_WARPS;
constexpr int TC_FEAT_THREADS = TC_FEAT_WARPS * 32;
constexpr int TC_MMA_WARP = TC_FEAT_WARPS;               // then the copy warp
constexpr int TC_COPY_WARP = TC_FEAT_WARPS + 1;
constexpr int TC_THREADS = TC_FEAT_THREADS + 64;
constexpr int TC_M = 128;         // keys per MMA block (= rows per ring tile)
constexpr int TC_N = 16;          // coefficient columns: hi and lo of up to eight heads
constexpr int TC_HEADS = TC_N / 2;
constexpr int TC_HSPLIT = TC_GROUP_WARPS / 4;          // warps sharing a quarter of the lanes
constexpr int TC_HPW = TC_HEADS / TC_HSPLIT;           // heads one read-out warp may hold
constexpr int TC_NBUF = 3;       // operand buffers and accumulators, used by block index mod 3
constexpr int TC_TMEM_COLS = 64;  // three accumulators of 16 columns (allocations are powers of two)
constexpr int TC_ROWS_PER_CTA = 16384;
constexpr int TC_PREFETCH = 6;  // tiles the copy warp prefetches into L2 ahead of the ring's newest
constexpr uint32_t TC_IDESC = f16_idesc(TC_M, TC_N);

template <int D>
struct TcGeo {
  static constexpr int F = D / 2;
  static constexpr int BPT = 4;                           // bf16 bands per lane (16 bytes)
  static constexpr int NP = BPT / 2;
  static constexpr int TPK = F / BPT;                     // lanes per key
  static constexpr int KPW = 32 / TPK;                    // keys per warp step
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int TILE_ROWS = TC_M;
  static constexpr int TILE_BYTES = TILE_ROWS * ROW_BYTES;
  static constexpr int NST = 65536 / TILE_BYTES;         // ring stages (64 KB)
  static constexpr int RPW = TILE_ROWS / TC_GROUP_WARPS;  // rows per warp per tile
  static constexpr int STEPS = RPW / KPW;                 // keys per lane per tile
  static constexpr int KF = 3 * F;                        // features per key
  static constexpr int KATOMS = (KF + 63) / 64;           // 64-feature columns of the operands
  static constexpr int KSTEPS = KF / 16;                  // MMAs per block (K = 16 each)
  static constexpr int A_ATOM = TC_M * 128;               // bytes of one column of A
  static constexpr int B_ATOM = TC_N * 128;
  static constexpr int A_BYTES = KATOMS * A_ATOM;
  static constexpr int B_BYTES = KATOMS * B_ATOM;
  static_assert(KF % 16 == 0 && STEPS >= 1 && RPW % KPW == 0 && NST >= 2, "geometry");
};

template <int NST>
struct TcCtrl {
  uint64_t full[NST];    // ring stage holds its tile (bulk copy completion)
  uint64_t empty[NST];   // a group is done with the stage's tile
  uint64_t a_full[TC_NBUF];    // per buffer: the features of its block are written
  uint64_t mma_done[TC_NBUF];  // per buffer: its block's MMAs have completed
  uint64_t d_free[TC_NBUF];    // per buffer: its accumulator was read out
  uint64_t final_done;   // every MMA issued has completed (exit)
  int failed;            // a wait timed out
  int issued;            // tiles whose copies were issued
  uint32_t tmem;         // accumulator base address
  int bad_block;
  uint32_t cmax[TC_HEADS];  // largest |coefficient| per head (float bits)
  float scale[TC_HEADS];    // power of two applied to the head's coefficients
  float unscale[TC_HEADS];  // its inverse
  // per band pair (re0, re1, im0, im1): e^{-i w k} for the step between a
  // lane's keys in a block and the jump to the group's next block
  float4 sstep[MAX_BANDS / 2], sjump[MAX_BANDS / 2];
};

template <int D>
struct TcLayout {
  using G = TcGeo<D>;
  static constexpr size_t OFF_A = 0;  // TC_NBUF operand buffers
  static constexpr size_t OFF_B = OFF_A + TC_NBUF * static_cast<size_t>(G::A_BYTES);
  static constexpr size_t OFF_RING = OFF_B + G::B_BYTES;
  static constexpr size_t OFF_CTRL = OFF_RING + static_cast<size_t>(G::NST) * G::TILE_BYTES;
  static constexpr size_t BYTES = OFF_CTRL + (sizeof(TcCtrl<G::NST>) + 15) / 16 * 16;
  static constexpr size_t SMEM = BYTES + 1024;  // room to align the operands to 1024 bytes
  static_assert(OFF_B % 1024 == 0 && OFF_RING % 1024 == 0, "operand alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  // statistics scratch [head][2][256] doubles, in A once the last MMA is done
  static_assert(TC_HEADS * 2 * 256 * sizeof(double) <= TC_NBUF * static_cast<size_t>(G::A_BYTES), "scratch fits");
  // coefficient scratch [TC_HEADS][F][3] floats, in A before the first block
  static_assert(TC_HEADS * G::F * 3 * sizeof(float) <= static_cast<size_t>(G::A_BYTES), "coefficients fit");
};

// Bulk prefetch of [p, p + bytes) into L2 (both 16-byte aligned): no shared
// memory, no completion to wait for.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  uint64_t ga;
  asm volatile("cvta.to.global.u64 %0, %1;" : "=l"(ga) : "l"(reinterpret_cast<uint64_t>(p)));
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ga), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int D, int STYLE, int PM>
__global__ void __launch_bounds__(TC_THREADS, 1)
    score_heads_tc_kernel(const __grid_constant__ ScoreParams p, int gh) {
  using T = uint16_t;
  using G = TcGeo<D>;
  using L = TcLayout<D>;
  constexpr bool EXPLICIT_POS = PM == POS_EXPLICIT, POST = PM == POS_POST_ROPE;
  constexpr int F = G::F, BPT = G::BPT, NP = G::NP, TPK = G::TPK, KPW = G::KPW, NST = G::NST;
  constexpr int ROW_BYTES = G::ROW_BYTES, TILE_ROWS = G::TILE_ROWS, RPW = G::RPW, STEPS = G::STEPS;

  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  unsigned char* sA = smem + L::OFF_A;
  unsigned char* sB = smem + L::OFF_B;
  unsigned char* ring = smem + L::OFF_RING;
  TcCtrl<NST>& ctrl = *reinterpret_cast<TcCtrl<NST>*>(smem + L::OFF_CTRL);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t s = blockIdx.x / p.tiles_per_slice;
  const int ct = blockIdx.x % p.tiles_per_slice;
  double* my_part = p.partials + ((s * p.tiles_per_slice + ct) * p.group + p.head0) * 3;

  const int n = p.n_valid[s];
  const bool bad = n > p.n_cap || n < 0;
  if (bad && tid == 0 && ct == 0) set_status(p.dev_status, TRI_DEV_NVALID_OVER_CAP);
  const int c0 = ct * p.rows_per_cta;
  const int c1 = bad ? c0 : min((ct + 1) * p.rows_per_cta, n);
  if (c0 >= c1) {  // nothing to score: empty partials (uniform over the CTA)
    if (tid < 3 * gh) my_part[tid] = 0.0;
    return;
  }
  const int ntiles = (c1 - c0 + TILE_ROWS - 1) / TILE_ROWS;  // = MMA blocks
  const unsigned char* kbase = static_cast<const unsigned char*>(p.k);
  const int64_t sbase = p.rows.slice_base(s);
  const int32_t* trow = p.rows.seq_table(s);
  if (!p.rows.blocks_ok(trow, c0, c1, &ctrl.bad_block)) {  // uniform over the CTA
    if (tid == 0) set_status(p.dev_status, TRI_DEV_BAD_BLOCK);
    if (tid < 3 * gh) my_part[tid] = 0.0;
    return;
  }

  if (tid == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(&ctrl.full[st], 1);
      mbar_init(&ctrl.empty[st], TC_GROUP_THREADS);
    }
    for (int b = 0; b < TC_NBUF; ++b) {
      mbar_init(&ctrl.a_full[b], TC_GROUP_THREADS);
      mbar_init(&ctrl.mma_done[b], 1);
      mbar_init(&ctrl.d_free[b], TC_GROUP_THREADS);
    }
    mbar_init(&ctrl.final_done, 1);
    ctrl.failed = 0;
    ctrl.issued = 0;
    mbar_init_fence();
  }
  if (tid < F / 2) {
    // e^{-i w_f x} for the lane's step between keys and its jump from one
    // block to the group's next, from the exact fixed-point phase
    const int f = 2 * tid;
    auto rot = [&](int x) {
      const float2 r0 = turns_rotation_accurate(-static_cast<int64_t>(x), p.nu[f]);
      const float2 r1 = turns_rotation_accurate(-static_cast<int64_t>(x), p.nu[f + 1]);
      return make_float4(r0.x, r1.x, r0.y, r1.y);
    };
    ctrl.sstep[tid] = rot(KPW);
    ctrl.sjump[tid] = rot(2 * TILE_ROWS - RPW);
  }
  if (tid < TC_HEADS) ctrl.cmax[tid] = 0u;
  if (warp == 0) {
    __syncwarp();  // the allocation is a whole-warp instruction
    tmem_alloc(&ctrl.tmem, TC_TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl.tmem;
  auto failed = [&]() { return *reinterpret_cast<volatile int*>(&ctrl.failed) != 0; };
  auto fail = [&]() { atomicExch(&ctrl.failed, 1); };
  // Named barrier 1 over every warp but the copy warp. The warp is
  // reconverged first, and the barrier form tolerates lanes that arrive
  // apart; the tensor-memory loads after barriers need whole warps.
  auto feat_sync = [&]() {
    __syncwarp();
    asm volatile("barrier.sync 1, %0;" ::"n"(TC_FEAT_THREADS + 32) : "memory");
  };

  const int lh = static_cast<int>(s % p.lh_count);
  const int64_t seq = s / p.lh_count;
  const int64_t pc = p.p_cur[seq];

  // ---- coefficient matrix B (once per CTA) ---------------------------------
  // The copy warp starts streaming right away; the others build B.
  float* cscr = reinterpret_cast<float*>(sA);
  if (warp != TC_COPY_WARP) {
    // pass 1: the heads' coefficients (Re W, Im W, n) into scratch in A, and
    // each head's largest magnitude
    for (int i = tid; i < gh * F; i += TC_FEAT_THREADS + 32) {
      const int g = i / F, f = i % F;
      const int64_t row = (static_cast<int64_t>(lh) * p.group + p.head0 + g) * F + f;
      const float2 cf = reinterpret_cast<const float2*>(p.center)[row];
      const float m = p.mean_norm[row];
      const float R = p.mrl[row];
      const float nw = (p.norm_mode == TRI_NORM_UNWEIGHTED) ? m : (1.0f - R) * m;
      float2 w = cmul(cf, make_float2(p.g_re[f], p.g_im[f]));
      if (POST) w = cmul(w, turns_rotation_accurate(pc, p.nu[f]));  // fold e^{i w p_cur} in
      cscr[i * 3 + 0] = w.x;
      cscr[i * 3 + 1] = w.y;
      cscr[i * 3 + 2] = nw;
      const float mx = fmaxf(fmaxf(fabsf(w.x), fabsf(w.y)), fabsf(nw));
      atomicMax(&ctrl.cmax[g], __float_as_uint(mx));  // non-negative floats order as their bits
    }
  }
  // ---- the copy warp: one thread streams the tiles through the ring -------
  // The ring holds one tile per group, which alone would leave the SM with
  // two tiles' bytes in flight from DRAM; tiles up to TC_PREFETCH beyond the
  // newest one in the ring are prefetched into L2, so the ring's own copies
  // mostly wait on L2 rather than DRAM.
  if (warp == TC_COPY_WARP) {
    if (lane == 0) {
      auto prefetch_tile = [&](int u) {
        const int r0 = c0 + u * TILE_ROWS;
        const int rows = min(TILE_ROWS, c1 - r0);
        for (int done = 0; done < rows;) {
          const int run = p.rows.run(r0 + done, rows - done);
          prefetch_l2(kbase + p.rows.row(sbase, trow, r0 + done), static_cast<uint32_t>(run * ROW_BYTES));
          done += run;
        }
      };
      for (int u = NST; u < min(ntiles, NST + TC_PREFETCH); ++u) prefetch_tile(u);
      for (int u = 0; u < ntiles; ++u) {
        const int st = u % NST;
        if (u >= NST && !mbar_wait_sleep(&ctrl.empty[st], static_cast<uint32_t>((u / NST - 1) & 1))) {
          fail();
          break;
        }
        if (failed()) break;
        const int r0 = c0 + u * TILE_ROWS;
        const int rows = min(TILE_ROWS, c1 - r0);
        uint64_t* bar = &ctrl.full[st];
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(rows * ROW_BYTES));
        unsigned char* dst = ring + st * G::TILE_BYTES;
        for (int done = 0; done < rows;) {
          const int run = p.rows.run(r0 + done, rows - done);
          bulk_g2s(dst + done * ROW_BYTES, kbase + p.rows.row(sbase, trow, r0 + done),
                   static_cast<uint32_t>(run * ROW_BYTES), bar);
          done += run;
        }
        ctrl.issued = u + 1;
        if (u >= NST && u + TC_PREFETCH < ntiles) prefetch_tile(u + TC_PREFETCH);
      }
    }
  } else {
    // named barrier over every warp but the copy warp: B is complete
    feat_sync();
    if (tid < TC_HEADS) {
      // 2^e with the head's largest coefficient in [2^13, 2^14)
      const uint32_t bits = ctrl.cmax[tid];
      const int ex = static_cast<int>((bits >> 23) & 0xffu) - 127;
      const int e = (bits == 0u || ex > 127) ? 0 : max(-100, min(100, 13 - ex));
      ctrl.scale[tid] = ldexpf(1.0f, e);
      ctrl.unscale[tid] = ldexpf(1.0f, -e);
    }
    feat_sync();
    // pass 2: B row nn = 2g (hi) or 2g + 1 (lo), feature k = section * F + f;
    // rows of absent heads and padding features are zero. Four features (8
    // bytes) per item.
    constexpr int KQ = G::KATOMS * 16;  // 4-feature pieces per row
    for (int i = tid; i < TC_N * KQ; i += TC_FEAT_THREADS + 32) {
      const int nn = i / KQ, k0 = (i % KQ) * 4;
      const int g = nn >> 1;
      uint32_t h[2] = {0u, 0u};
      if (g < gh && k0 < G::KF) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = k0 + e;
          const int sec = k / F, f = k % F;
          const float x = cscr[(g * F + f) * 3 + sec] * ctrl.scale[g];
          const float hi = __half2float(__float2half_rn(x));
          v[e] = (nn & 1) ? x - hi : hi;
        }
        h[0] = pack_half2(v[0], v[1]);
        h[1] = pack_half2(v[2], v[3]);
      }
      const int atom = k0 / 64, b = (k0 % 64) * 2;
      *reinterpret_cast<uint2*>(sB + atom * G::B_ATOM + sw128_offset(nn, b)) = make_uint2(h[0], h[1]);
    }
    fence_proxy_async_smem();  // B is read by the tensor cores
    feat_sync();  // and A is free again
  }

  float sh[TC_HPW] = {}, s1[TC_HPW] = {}, s2[TC_HPW] = {};
  int cnt = 0;
  int mma_issued = 0;  // MMA thread: blocks issued
  const int hpw = (gh + TC_HSPLIT - 1) / TC_HSPLIT;  // heads per read-out warp
  if (warp == TC_MMA_WARP) {
    // ---- the MMA warp: the whole warp follows the blocks (its values stay
    // warp-uniform); one elected lane issues every block's MMAs -------------
    const uint64_t b_desc0 = sw128_desc(smem_addr(sB));
    const uint64_t a_desc0 = sw128_desc(smem_addr(sA));
    for (int t = 0; t < ntiles; ++t) {
      // block t uses operand buffer and accumulator bi; accumulator bi is
      // free once block t - 3 was read out
      const int bi = t % TC_NBUF;
      bool ok = mbar_wait_backoff(&ctrl.a_full[bi], static_cast<uint32_t>((t / TC_NBUF) & 1));
      if (ok && t >= TC_NBUF)
        ok = mbar_wait_backoff(&ctrl.d_free[bi], static_cast<uint32_t>((t / TC_NBUF - 1) & 1));
      ok = __all_sync(FULL_MASK, ok) && !failed();
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + static_cast<uint32_t>(bi * TC_N);
      const uint64_t a_desc = a_desc0 + ((static_cast<uint64_t>(bi) * G::A_BYTES) >> 4);
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < G::KSTEPS; ++k) {
          // descriptor start addresses advance in 16-byte units
          const uint64_t off_a = ((k / 4) * G::A_ATOM + (k % 4) * 32) >> 4;
          const uint64_t off_b = ((k / 4) * G::B_ATOM + (k % 4) * 32) >> 4;
          umma_f16(d, a_desc + off_a, b_desc0 + off_b, TC_IDESC, k > 0);
        }
        umma_commit(&ctrl.mma_done[bi]);
      }
      __syncwarp();
      mma_issued = t + 1;
    }
  } else if (warp < TC_FEAT_WARPS) {
    // ---- the feature warps: group gi takes tiles gi, gi + 2, ... -----------
    const int gi = warp / TC_GROUP_WARPS, gw = warp % TC_GROUP_WARPS;
    const int c = lane % TPK;
    const int kq = lane / TPK;
    const int rbase = gw * RPW + kq;  // this lane's first row in a tile
    float2 ER[NP], EI[NP], SR[NP], SI[NP], NSI[NP];
    uint64_t nu[BPT];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      float er[2] = {1.f, 1.f}, ei[2] = {0.f, 0.f};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int f = c * BPT + 2 * q + hh;
        nu[2 * q + hh] = p.nu[f];
        if (PM == POS_SLOT) {
          const float2 e = turns_rotation_accurate(pc - (c0 + gi * TILE_ROWS + rbase), p.nu[f]);
          er[hh] = e.x;
          ei[hh] = e.y;
        }
      }
      const int f0 = c * BPT + 2 * q;
      ER[q] = f2(er[0], er[1]);
      EI[q] = f2(ei[0], ei[1]);
      const float4 sq4 = ctrl.sstep[f0 / 2];
      SR[q] = f2(sq4.x, sq4.y);
      SI[q] = f2(sq4.z, sq4.w);
      NSI[q] = f2(-sq4.z, -sq4.w);
    }
    // where this lane's three 8-byte feature pieces of its j-th key go in A
    // (row rbase + j*KPW of the block)
    uint32_t aoff[STEPS][3];
#pragma unroll
    for (int j = 0; j < STEPS; ++j) {
#pragma unroll
      for (int sec = 0; sec < 3; ++sec) {
        const int k = sec * F + c * BPT;
        aoff[j][sec] = static_cast<uint32_t>((k / 64) * G::A_ATOM) + sw128_offset(rbase + j * KPW, (k % 64) * 2);
      }
    }

    float* out = p.scores_g + (s * p.group + p.head0) * static_cast<int64_t>(p.n_cap);
    const int32_t* pos = EXPLICIT_POS ? p.pos + s * static_cast<int64_t>(p.n_cap) : nullptr;
    // read-out role: lanes 32*eq .. of the accumulator, heads eg .. eg+hpw-1
    const int eq = gw & 3, eg = (gw >> 2) * hpw;

    // a wait by the whole warp (uniform result; the warp is converged after it)
    auto warp_wait = [&](uint64_t* bar, int phase) {
      bool w = mbar_wait_sleep(bar, static_cast<uint32_t>(phase & 1));
      w = __all_sync(FULL_MASK, w);
      if (!w && lane == 0) fail();
      return w;
    };
    // the scores of block b (this group's) from its accumulator
    auto readout = [&](int b) {
      const int bi = b % TC_NBUF;
      if (!warp_wait(&ctrl.mma_done[bi], b / TC_NBUF)) return false;
      tc_fence_after();
      if (eg < gh) {  // warp-uniform
        uint32_t d[2 * TC_HPW];
        __syncwarp();  // the load is a whole-warp (aligned) instruction
        const uint32_t ta = tmem + (static_cast<uint32_t>(eq * 32) << 16) + static_cast<uint32_t>(bi * TC_N + 2 * eg);
        tmem_ld8(ta, *reinterpret_cast<uint32_t(*)[8]>(&d[0]));
        if constexpr (TC_HPW > 4) {
          if (hpw > 4) tmem_ld8(ta + 8u, *reinterpret_cast<uint32_t(*)[8]>(&d[8]));
        }
        tmem_wait_ld();
        const int row = c0 + b * TC_M + eq * 32 + lane;
        if (row < c1) {
#pragma unroll
          for (int h = 0; h < TC_HPW; ++h) {
            const int g = eg + h;
            if (h < hpw && g < gh) {
              const float v = (__uint_as_float(d[2 * h]) + __uint_as_float(d[2 * h + 1])) * ctrl.unscale[g];
              __stcs(out + static_cast<int64_t>(g) * p.n_cap + row, v);
              if (cnt == 0) sh[h] = v;
              const float dv = v - sh[h];
              s1[h] += dv;
              s2[h] = fmaf(dv, dv, s2[h]);
            }
          }
          ++cnt;
        }
      }
      tc_fence_before();
      mbar_arrive(&ctrl.d_free[bi]);
      return true;
    };

    int last = -1;  // this group's last block
    for (int t = gi; t < ntiles; t += 2) {
      if (!warp_wait(&ctrl.full[t % NST], t / NST)) break;
      // the lane's chunks of the tile go to registers, and the stage is
      // handed back to the copy warp before any arithmetic
      const unsigned char* tile = ring + (t % NST) * G::TILE_BYTES;
      uint4 raw[STEPS];
#pragma unroll
      for (int j = 0; j < STEPS; ++j) raw[j] = lds_chunk<T, D, STYLE>(tile + (rbase + j * KPW) * ROW_BYTES, c);
      mbar_arrive(&ctrl.empty[t % NST]);
      // operand buffer t % 3 held block t - 3 (the other group's): free once
      // that block's MMAs are done
      if (t >= TC_NBUF && !warp_wait(&ctrl.mma_done[t % TC_NBUF], t / TC_NBUF - 1)) break;
      unsigned char* a = sA + (t % TC_NBUF) * G::A_BYTES;
      int pp[STEPS];
      if (EXPLICIT_POS) {
#pragma unroll
        for (int j = 0; j < STEPS; ++j) {
          const int r = c0 + t * TILE_ROWS + rbase + j * KPW;
          pp[j] = (r < c1) ? __ldg(pos + r) : 0;
        }
      }
#pragma unroll
      for (int j = 0; j < STEPS; ++j) {
        // rows past the run's end hold stale bytes: their accumulator rows
        // are never read out
        float re[BPT], im[BPT];
        decode_chunk<T, STYLE>(raw[j], re, im);
        uint32_t hz[NP], hn[NP], hm[NP];
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          const float2 RE = f2(re[2 * q], re[2 * q + 1]);
          const float2 IM = f2(im[2 * q], im[2 * q + 1]);
          const float2 sq = __ffma2_rn(IM, IM, __fmul2_rn(RE, RE));
          hm[q] = pack_half2(sqrt_approx(sq.x), sqrt_approx(sq.y));
          if (POST) {
            hz[q] = pack_half2(RE.x, RE.y);
            hn[q] = pack_half2(IM.x, IM.y);
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
          hz[q] = pack_half2(zr.x, zr.y);
          hn[q] = pack_half2(zn.x, zn.y);
        }
        *reinterpret_cast<uint2*>(a + aoff[j][0]) = make_uint2(hz[0], hz[1]);
        *reinterpret_cast<uint2*>(a + aoff[j][1]) = make_uint2(hn[0], hn[1]);
        *reinterpret_cast<uint2*>(a + aoff[j][2]) = make_uint2(hm[0], hm[1]);
      }
      fence_proxy_async_smem();  // the features are read by the tensor cores
      mbar_arrive(&ctrl.a_full[t % TC_NBUF]);
      // the group's previous block, whose MMAs ran while these features
      // were formed
      if (t >= 2 && !readout(t - 2)) break;
      last = t;
      if (failed()) break;
      if (PM == POS_SLOT) {
        // from this lane's last key of tile t to its first key of tile t + 2
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          const float4 jq = ctrl.sjump[c * NP + q];
          const float2 jr = f2(jq.x, jq.y), ji = f2(jq.z, jq.w), nji = f2(-jq.z, -jq.w);
          const float2 er = ER[q], ei = EI[q];
          ER[q] = __ffma2_rn(er, jr, __fmul2_rn(ei, nji));
          EI[q] = __ffma2_rn(er, ji, __fmul2_rn(ei, jr));
        }
      }
    }
    if (last >= 0 && !failed()) readout(last);
  }

  // ---- exit: every copy landed and every MMA completed before the shared and
  // tensor memory go ---------------------------------------------------------
  __syncwarp();  // the copy warp's lanes meet again
  __syncthreads();
  if (warp == TC_MMA_WARP && mma_issued > 0) {
    if (elect_one()) umma_commit(&ctrl.final_done);  // arrives once every earlier MMA of that lane is done
    __syncwarp();
    if (!mbar_wait_bounded(&ctrl.final_done, 0u) && lane == 0) fail();
  }
  if (warp == TC_COPY_WARP && lane == 0 && failed()) {
    set_status(p.dev_status, TRI_DEV_TIMEOUT);
    const int is = ctrl.issued;
    for (int u = max(0, is - NST); u < is; ++u)
      (void)mbar_wait_bounded(&ctrl.full[u % NST], static_cast<uint32_t>((u / NST) & 1));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TC_TMEM_COLS);
  }

  // ---- statistics partials of this CTA, per head, in fp64 -------------------
  // Head g was read out by the 256 threads of both groups' warps with
  // gw / 4 == g / hpw, slot g % hpw; each turns its shifted sums into plain
  // ones, and a tree of fixed shape adds the 256 (the fp64 pipe is slow, so
  // no long serial chain). Every row of the run was read once per head: the
  // count is c1 - c0.
  double* spart = reinterpret_cast<double*>(sA);  // [head][sum, sum of squares][256]
  if (tid < TC_FEAT_THREADS) {
    const int gw = warp % TC_GROUP_WARPS, half = gw >> 2;
    const int ci = ((warp / TC_GROUP_WARPS) * 4 + (gw & 3)) * 32 + lane;
    const double dn = cnt;
#pragma unroll
    for (int h = 0; h < TC_HPW; ++h) {
      const int g = half * hpw + h;
      if (h < hpw && g < gh) {
        const double dsh = sh[h], ds1 = s1[h];
        spart[(g * 2 + 0) * 256 + ci] = dn * dsh + ds1;
        spart[(g * 2 + 1) * 256 + ci] = dn * dsh * dsh + 2.0 * dsh * ds1 + static_cast<double>(s2[h]);
      }
    }
  }
  __syncthreads();
  for (int stride = 128; stride >= 1; stride >>= 1) {
    for (int i = tid; i < gh * 2 * stride; i += TC_THREADS) {
      const int gv = i / stride, k = i % stride;
      spart[gv * 256 + k] += spart[gv * 256 + k + stride];
    }
    __syncthreads();
  }
  if (tid < gh) {
    my_part[3 * tid + 0] = spart[(tid * 2 + 0) * 256];
    my_part[3 * tid + 1] = spart[(tid * 2 + 1) * 256];
    my_part[3 * tid + 2] = static_cast<double>(c1 - c0);
  }
}

template <int D, int STYLE, int PM>
cudaError_t launch_tc(const ScoreParams& p, int n_heads, int n_slices, cudaStream_t st) {
  auto kern = score_heads_tc_kernel<D, STYLE, PM>;
  const size_t smem = TcLayout<D>::SMEM;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(n_slices) * p.tiles_per_slice));
  kern<<<grid, TC_THREADS, smem, st>>>(p, n_heads);
  note_launch();
  return cudaGetLastError();
}

template <int D, int STYLE>
cudaError_t launch_tc_pm(const ScoreParams& p, int n_heads, int pm, int n_slices, cudaStream_t st) {
  if (pm == POS_POST_ROPE) return launch_tc<D, STYLE, POS_POST_ROPE>(p, n_heads, n_slices, st);
  if (pm == POS_EXPLICIT) return launch_tc<D, STYLE, POS_EXPLICIT>(p, n_heads, n_slices, st);
  return launch_tc<D, STYLE, POS_SLOT>(p, n_heads, n_slices, st);
}

template <int D>
ScoreGeometry tc_geo() {
  using G = TcGeo<D>;
  // a lane's keys within a block are KPW apart; from its last key of block t
  // (one step already taken) to its first key of block t + 2 (the kernel
  // forms both rotations itself); runs are whole blocks
  return ScoreGeometry{G::KPW, 2 * G::TILE_ROWS - G::RPW, G::TILE_ROWS};
}

}  // namespace

ScoreGeometry tc_heads_geometry(int head_dim, int32_t& max_rows_per_cta) {
  max_rows_per_cta = TC_ROWS_PER_CTA;
  return head_dim == 128 ? tc_geo<128>() : tc_geo<64>();
}

cudaError_t launch_score_heads_tc(const ScoreParams& p, int n_heads, int head_dim, tri_rope_style style,
                                  int pos_mode, int n_slices, cudaStream_t st) {
  if (n_heads < 1 || n_heads > TC_HEADS) return cudaErrorInvalidValue;
  if (p.rows_per_cta % TC_M != 0) return cudaErrorInvalidValue;
  if (head_dim == 128) {
    return style == TRI_ROPE_INTERLEAVED ? launch_tc_pm<128, TRI_ROPE_INTERLEAVED>(p, n_heads, pos_mode, n_slices, st)
                                         : launch_tc_pm<128, TRI_ROPE_HALF>(p, n_heads, pos_mode, n_slices, st);
  }
  return style == TRI_ROPE_INTERLEAVED ? launch_tc_pm<64, TRI_ROPE_INTERLEAVED>(p, n_heads, pos_mode, n_slices, st)
                                       : launch_tc_pm<64, TRI_ROPE_HALF>(p, n_heads, pos_mode, n_slices, st);
}

}  // namespace tri
