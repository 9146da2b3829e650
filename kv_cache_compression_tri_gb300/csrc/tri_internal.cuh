// tri_internal.cuh -- device helpers and launcher declarations shared by the
// kernels of libtri (GPU side only; the oracle has its own code).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/tri.h"

namespace tri {

constexpr unsigned FULL_MASK = 0xffffffffu;
constexpr int MAX_BANDS = 64;  // head_dim <= 128

// Count of kernels launched by the library (tri_launch_count).
void note_launch();

// An NVTX range named after the entry point, open for the call's host-side
// part (argument checks and launches): a profiler that records NVTX shows
// every library call on its timeline, named; without one the NVTX calls do
// nothing (header-only NVTX v3, no library to link).
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};
#define TRI_CALL_RANGE() const ::tri::CallRange tri_call_range_(__func__)

// First error wins: a device status word goes from 0 to `code` once.
__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}

// bf16 halves of a 32-bit word as fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// e^{i 2 pi frac(x * nu)} where nu is a 0.64 fixed-point number of turns per
// position: the product is exact mod 2^64, so the phase keeps full precision
// at any position. Accurate variant (sincospif), for anchors.
__device__ __forceinline__ float2 turns_rotation_accurate(int64_t x, uint64_t nu) {
  const uint64_t t = static_cast<uint64_t>(x) * nu;  // wraps mod 2^64
  // signed turns in [-0.5, 0.5) -> argument of sincospi in [-1, 1)
  const float a = static_cast<float>(static_cast<int64_t>(t)) * 1.0842021724855044e-19f;  // 2^-63
  float s, c;
  sincospif(a, &s, &c);
  return make_float2(c, s);
}

// Fast variant (hardware sin/cos on an argument already reduced to
// [-pi, pi)), for per-key rotations. x must lie in [0, 2^32) (a key's age):
// the top 32 bits of the phase x * nu (mod 2^64) are then exactly
// hi32(x * nu_lo) + x * nu_hi (mod 2^32), two 32-bit multiplies.
__device__ __forceinline__ float2 turns_rotation_fast(int64_t x, uint64_t nu) {
  const uint32_t x32 = static_cast<uint32_t>(x);
  const uint32_t top = __umulhi(x32, static_cast<uint32_t>(nu)) + x32 * static_cast<uint32_t>(nu >> 32);
  const int32_t hi = static_cast<int32_t>(top);
  const float ang = static_cast<float>(hi) * 1.4629180792671596e-09f;  // 2 pi / 2^32
  float s, c;
  __sincosf(ang, &s, &c);
  return make_float2(c, s);
}

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
  return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}

// Philox-4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11): per round
// two 32x32->64 multiplies feed the next (x0..x3); the key is bumped by the
// Weyl increments between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 x, uint2 key) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      key.x += 0x9E3779B9u;
      key.y += 0xBB67AE85u;
    }
    const uint32_t m0 = 0xD2511F53u, m1 = 0xCD9E8D57u;
    const uint32_t hi0 = __umulhi(m0, x.x), lo0 = m0 * x.x;
    const uint32_t hi1 = __umulhi(m1, x.z), lo1 = m1 * x.z;
    x = make_uint4(hi1 ^ x.y ^ key.x, lo1, hi0 ^ x.w ^ key.y, lo0);
  }
  return x;
}

// ---------------------------------------------------------------------------
// Bulk async copies (TMA, non-tensor) into shared memory with mbarrier
// completion, and a wall-clock-bounded wait.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// Order this thread's earlier shared-memory accesses before later async-proxy
// writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned); completion is counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  uint64_t gsrc;
  asm volatile("cvta.to.global.u64 %0, %1;" : "=l"(gsrc) : "l"(src));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// shared -> global bulk copy (same alignment rules), tracked as a bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  uint64_t gdst;
  asm volatile("cvta.to.global.u64 %0, %1;" : "=l"(gdst) : "l"(dst));
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar`; gives up after ~2 s of wall clock so a
// lost completion can never hang the GPU (the caller reports TRI_DEV_TIMEOUT).
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
__device__ __forceinline__ bool mbar_wait_limit(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  return mbar_wait_limit(bar, parity, WAIT_LIMIT_NS);
}

// sqrt of a non-negative fp32 (hardware approximation; exact at 0). The
// flush-to-zero form: a subnormal input (a band of squared magnitude below
// 2^-126) reads as 0, which leaves no trace at the score tolerance, and the
// instruction needs none of the subnormal handling of the IEEE form.
__device__ __forceinline__ float sqrt_approx(float x) {
  float r;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Order-preserving map of an fp32 score to u32 (larger score -> larger key).
// -0 is folded onto +0; NaN maps to 0 (below every number) and is flagged.
__device__ __forceinline__ uint32_t score_key(float x, bool& nan) {
  if (x != x) {
    nan = true;
    return 0u;
  }
  uint32_t u = __float_as_uint(x);
  if (x == 0.0f) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// z-score of one query head's score, from the head's mean and 1/std over the
// slice (TriAttention paper summary, "Handling Grouped-Query Attention"); a
// head whose scores are all equal (std 0) gives 0. Every kernel that ranks or
// reports z-scores uses these two, so they agree bit for bit.
__device__ __forceinline__ float head_inv_std(float sd) { return sd > 0.f ? 1.0f / sd : 0.f; }
__device__ __forceinline__ float head_z(float v, float mu, float inv) { return __fmul_rn(__fsub_rn(v, mu), inv); }

// Where the K (or V) row r of slice s lives: contiguous slices at a uniform
// stride, or a paged pool addressed through the sequence's block table.
struct RowMap {
  int64_t slice_bytes;   // contiguous: bytes between slices
  const int32_t* table;  // paged: [n_seq][max_blocks]; NULL for contiguous slices
  int32_t block_size, block_shift, max_blocks, num_blocks;  // block_size = 1 << block_shift
  int64_t block_bytes, layer_bytes, head_bytes;
  int32_t lh_count, n_kv_heads, row_bytes;

  __device__ __forceinline__ bool paged() const { return table != nullptr; }
  // byte offset of the slice's row 0 (paged: within block 0 of the pool)
  __device__ __forceinline__ int64_t slice_base(int64_t s) const {
    if (!table) return s * slice_bytes;
    const int64_t lh = s % lh_count;
    return (lh / n_kv_heads) * layer_bytes + (lh % n_kv_heads) * head_bytes;
  }
  __device__ __forceinline__ const int32_t* seq_table(int64_t s) const {
    return table ? table + (s / lh_count) * static_cast<int64_t>(max_blocks) : nullptr;
  }
  // byte offset of row r, given slice_base and seq_table of its slice
  __device__ __forceinline__ int64_t row(int64_t base, const int32_t* trow, int r) const {
    if (!table) return base + static_cast<int64_t>(r) * row_bytes;
    return base + static_cast<int64_t>(__ldg(trow + (r >> block_shift))) * block_bytes +
           static_cast<int64_t>(r & (block_size - 1)) * row_bytes;
  }
  // rows r, r+1, ... that are contiguous in memory (at most `limit`)
  __device__ __forceinline__ int run(int r, int limit) const {
    return table ? min(limit, block_size - (r & (block_size - 1))) : limit;
  }
  // every table entry for rows [r0, r1) lies in [0, num_blocks) (by the CTA;
  // uniform result). When `cache` is given, the entries of blocks cache_b0 ..
  // cache_b0 + cache_n - 1 among them are kept there (cache_b0 < 0: from the
  // block of row r0; by default every entry checked).
  __device__ __forceinline__ bool blocks_ok(const int32_t* trow, int r0, int r1, int* sflag,
                                            int32_t* cache = nullptr, int cache_b0 = -1,
                                            int cache_n = 0x7fffffff) const {
    if (!table || r0 >= r1) return true;
    if (threadIdx.x == 0) *sflag = 0;
    __syncthreads();
    const int b0 = r0 >> block_shift;
    const int cb0 = cache_b0 < 0 ? b0 : cache_b0;
    for (int b = b0 + static_cast<int>(threadIdx.x); b <= ((r1 - 1) >> block_shift); b += static_cast<int>(blockDim.x)) {
      const int v = __ldg(trow + b);
      if (v < 0 || v >= num_blocks) *sflag = 1;
      if (cache && b >= cb0 && b - cb0 < cache_n) cache[b - cb0] = v;
    }
    __syncthreads();
    const bool ok = *sflag == 0;
    __syncthreads();
    return ok;
  }
};

// ---------------------------------------------------------------------------
// Kernel parameter blocks (passed by value).
// ---------------------------------------------------------------------------
struct ScoreParams {
  const void* k;
  const int32_t* pos;
  const int32_t* n_valid;
  const int64_t* p_cur;
  const float* center;
  const float* mean_norm;
  const float* mrl;
  float* scores;
  int32_t* dev_status;
  RowMap rows;  // where the K rows are
  int32_t n_cap;
  int32_t lh_count;  // n_layers * n_kv_heads
  int32_t n_prompt, n_recent;
  int32_t norm_mode;
  int32_t tiles_per_slice;  // CTAs per slice
  int32_t rows_per_cta;
  uint64_t nu[MAX_BANDS];     // omega_f / 2pi as 0.64 fixed point (turns per position)
  float g_re[MAX_BANDS];      // G_f = (1/|D|) sum_delta e^{i omega_f delta}
  float g_im[MAX_BANDS];
  float step_re[MAX_BANDS];   // e^{-i omega_f * (positions between a lane's keys in a tile)}
  float step_im[MAX_BANDS];
  float jump_re[MAX_BANDS];   // e^{-i omega_f * (positions skipped between tiles)}
  float jump_im[MAX_BANDS];
  // per-query-head scoring (GQA): centre rows are (layer * H + h) * group + g
  int32_t group;     // query heads per KV head
  int32_t head0;     // first query head (within the group) of this launch
  float* scores_g;   // [S][group][n_cap]
  double* partials;  // [S][tiles_per_slice][group][3]: sum, sum of squares, rows
};

struct SelectParams {
  const float* scores;  // [S][n_cap] (score source)
  const int32_t* n_valid;
  int32_t* keep;  // [S][budget]
  int32_t* dev_status;
  int32_t n_cap, n_prompt, n_recent, budget;
  int32_t n_layers, n_kv_heads;
  uint64_t seed;
  uint32_t round;
  int32_t draw_scope;  // 0: a draw per KV head; 1: one per (seq, layer); 2: one per sequence
  // z-score + max source: per-head scores [S][group][n_cap], stats [S][group][2]
  const float* stats;
  int32_t group;
  // union source: per-group union bitmap [groups][member_words], member counts [groups]
  const uint32_t* member;
  const int32_t* ucount;
  int32_t member_words;
};

struct UnionPrepParams {
  const float* scores;    // [S][n_cap], every valid row scored
  const int32_t* n_valid;
  const int32_t* keepk;   // [S][bk]: each slice's own top picks (or NULL when bk == 0)
  uint32_t* member;       // [groups][member_words] out
  int32_t* ucount;        // [groups] out
  int32_t* dev_status;
  int32_t n_cap, bk, n_prompt, n_recent, group, member_words;
};

struct CompactParams {
  char* k;
  char* v;
  const int32_t* pos;
  int32_t* pos_out;
  int32_t* n_valid;
  const int32_t* keep;
  int32_t* dev_status;
  RowMap rows;  // where the K and V rows are (same layout for both)
  int32_t n_cap;
  int32_t budget;
  int32_t row_bytes;
};

struct CalibParams {
  const void* q;
  float* ws;
  float* center;
  float* mean_norm;
  float* mrl;
  int32_t n_q_heads, group, n_split;
  int32_t kv_heads;
  int64_t n_tok;
};

// Launchers (return cudaSuccess or the launch error).
// pos_mode: 0 pre-RoPE keys at their slot index, 1 pre-RoPE keys with a
// position array, 2 post-RoPE keys (positions unused).
cudaError_t launch_score(const ScoreParams& p, tri_dtype dt, int head_dim, tri_rope_style style,
                         int pos_mode, int n_slices, cudaStream_t st);
// Score kernel geometry, shared by the launcher and the host constant table:
// positions between consecutive keys of one lane inside a tile, and the
// positions skipped from a lane's last key of a tile to its first of the next.
struct ScoreGeometry {
  int step;
  int jump;
  int tile_rows;
};
ScoreGeometry score_geometry(tri_dtype dt, int head_dim);
cudaError_t launch_select(const SelectParams& p, int n_slices, cudaStream_t st);
// Score (rows [P, n - W)), selection and compaction of every slice in one
// launch, one CTA per slice; requires p.tiles_per_slice == 1.
cudaError_t launch_compress_slices(const ScoreParams& p, const SelectParams& ps, const CompactParams& pc,
                                   tri_dtype dt, int head_dim, tri_rope_style style, int pos_mode, int n_slices,
                                   cudaStream_t st);
// Per-query-head scores and per-CTA statistics partials, heads [head0, head0 +
// n_heads) of every group; then the per-(slice, head) mean and standard
// deviation; then (optional) the z-score maximum of every valid row.
// fp32 keys: CUDA-core kernel, up to four heads per launch; bf16 keys: the
// heads' contraction on the tensor cores, up to eight heads per launch.
constexpr int MAX_HEADS_PER_LAUNCH = 4;
constexpr int MAX_HEADS_PER_LAUNCH_TC = 8;
constexpr int MAX_GROUP = 8;
cudaError_t launch_score_heads(const ScoreParams& p, int n_heads, tri_dtype dt, int head_dim,
                               tri_rope_style style, int pos_mode, int n_slices, cudaStream_t st);
cudaError_t launch_score_heads_tc(const ScoreParams& p, int n_heads, int head_dim, tri_rope_style style,
                                  int pos_mode, int n_slices, cudaStream_t st);
// lane geometry (step, jump, rows per tile) of the tensor-core kernel and its
// largest run of rows per CTA
ScoreGeometry tc_heads_geometry(int head_dim, int32_t& max_rows_per_cta);
cudaError_t launch_heads_stats(const double* partials, float* stats, int n_slices, int tiles_per_slice,
                               int group, cudaStream_t st);
// out[b][i] = max_g z of rows [b*group, b*group+group) for blocks b < n_blocks;
// the valid row count of block b is n_valid[b * nv_stride].
cudaError_t launch_zmax_scores(const float* scores_g, const float* stats, const int32_t* n_valid, int nv_stride,
                               float* out, int n_blocks, int n_cap, int group, cudaStream_t st);
cudaError_t launch_union_prep(const UnionPrepParams& q, int n_groups, cudaStream_t st);
cudaError_t launch_slice_stats(const float* scores, const int32_t* n_valid, float* stats, int n_slices, int n_cap,
                               cudaStream_t st);
cudaError_t launch_blocks_used(const RowMap& rows, const int32_t* n_valid, int32_t* blocks_used, int n_seq,
                               cudaStream_t st);
// Self-test of the bounded waits: one thread waits on an mbarrier that
// nothing arrives on, for at most limit_ns, and records TRI_DEV_TIMEOUT.
cudaError_t launch_wait_timeout_selftest(int32_t* dev_status, uint64_t limit_ns, cudaStream_t st);
cudaError_t launch_select_union(const SelectParams& p, int n_groups, cudaStream_t st);
cudaError_t launch_select_zmax(const SelectParams& p, int n_slices, cudaStream_t st);
cudaError_t launch_rand_select(const SelectParams& p, int n_slices, cudaStream_t st);
cudaError_t launch_compact(const CompactParams& p, int n_slices, cudaStream_t st);
// Selection (by score, or by Random Attention draw when `random`) then
// compaction of each slice in one CTA.
cudaError_t launch_select_compact(const SelectParams& ps, const CompactParams& pc, bool random, int n_slices,
                                  cudaStream_t st);
cudaError_t launch_calibrate(const CalibParams& p, tri_dtype dt, int head_dim,
                             tri_rope_style style, int lh_count, cudaStream_t st);
int calibrate_split_count(int lh_count, int64_t samples_per_lh);

}  // namespace tri
