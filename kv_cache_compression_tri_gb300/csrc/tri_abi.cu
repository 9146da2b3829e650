// tri_abi.cu -- the extern "C" entry points of libtri (include/tri.h).
//
// Each entry point validates its arguments on the host, fills a kernel
// parameter block, and enqueues its kernels on the caller's stream. Nothing
// here allocates device memory or synchronises. The only host arithmetic is
// the per-band constant table of tri_score (at most 64 bands x 5 numbers,
// from rope_theta and the offset set), computed in fp64.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "tri_internal.cuh"

namespace tri {

static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_bytes(tri_dtype dt) { return dt == TRI_BF16 ? 2 : 4; }

// Shape checks shared by every call that takes a tri_kv.
tri_status check_kv(const tri_kv* kv, bool need_v) {
  if (!kv) return TRI_ERR_INVALID_ARG;
  if (kv->dtype != TRI_BF16 && kv->dtype != TRI_F32) return TRI_ERR_UNSUPPORTED;
  if (kv->head_dim != 64 && kv->head_dim != 128) return TRI_ERR_UNSUPPORTED;
  if (kv->n_seq < 1 || kv->n_layers < 1 || kv->n_kv_heads < 1 || kv->n_cap < 1)
    return TRI_ERR_INVALID_ARG;
  const int64_t n_slices = static_cast<int64_t>(kv->n_seq) * kv->n_layers * kv->n_kv_heads;
  if (n_slices > 0x7fffffff) return TRI_ERR_INVALID_ARG;
  if (!kv->n_valid || !aligned(kv->n_valid, 4)) return TRI_ERR_INVALID_ARG;
  if (!kv->k || !aligned(kv->k, 16)) return TRI_ERR_INVALID_ARG;
  if (need_v && (!kv->v || !aligned(kv->v, 16))) return TRI_ERR_INVALID_ARG;
  const int e = elem_bytes(kv->dtype);
  if (kv->block_table) {
    // paged pools: whole blocks of 16-byte aligned rows
    if (!aligned(kv->block_table, 4)) return TRI_ERR_INVALID_ARG;
    const int bsz = kv->block_size;
    if (bsz < 16 || (bsz & (bsz - 1)) != 0 || kv->n_cap % bsz != 0) return TRI_ERR_INVALID_ARG;  // a power of two
    if (kv->num_blocks < 1) return TRI_ERR_INVALID_ARG;
    for (const int64_t st : {kv->block_stride, kv->layer_stride, kv->head_stride})
      if (st < 0 || (st * e) % 16 != 0) return TRI_ERR_INVALID_ARG;
    if (kv->head_stride < static_cast<int64_t>(kv->block_size) * kv->head_dim) return TRI_ERR_INVALID_ARG;
  } else {
    if (kv->slice_stride < static_cast<int64_t>(kv->n_cap) * kv->head_dim) return TRI_ERR_INVALID_ARG;
    if ((kv->slice_stride * e) % 16 != 0) return TRI_ERR_INVALID_ARG;
  }
  if (kv->pos && !aligned(kv->pos, 4)) return TRI_ERR_INVALID_ARG;
  if (kv->pos_out && !aligned(kv->pos_out, 4)) return TRI_ERR_INVALID_ARG;
  if (kv->dev_status && !aligned(kv->dev_status, 4)) return TRI_ERR_INVALID_ARG;
  if (kv->key_layout != TRI_KEYS_PRE_ROPE && kv->key_layout != TRI_KEYS_POST_ROPE) return TRI_ERR_INVALID_ARG;
  return TRI_OK;
}

// Row addressing of the cache for the kernels.
RowMap row_map(const tri_kv* kv) {
  RowMap m{};
  const int e = elem_bytes(kv->dtype);
  m.row_bytes = kv->head_dim * e;
  m.lh_count = kv->n_layers * kv->n_kv_heads;
  m.n_kv_heads = kv->n_kv_heads;
  if (kv->block_table) {
    m.table = kv->block_table;
    m.block_size = kv->block_size;
    m.block_shift = __builtin_ctz(static_cast<unsigned>(kv->block_size));
    m.max_blocks = kv->n_cap / kv->block_size;
    m.num_blocks = kv->num_blocks;
    m.block_bytes = kv->block_stride * e;
    m.layer_bytes = kv->layer_stride * e;
    m.head_bytes = kv->head_stride * e;
  } else {
    m.slice_bytes = kv->slice_stride * e;
  }
  return m;
}

// Where the score kernels take each key's rotation from (see launch_score).
int pos_mode(const tri_kv* kv) {
  if (kv->key_layout == TRI_KEYS_POST_ROPE) return 2;
  return kv->pos ? 1 : 0;
}

int64_t slices_of(const tri_kv* kv) {
  return static_cast<int64_t>(kv->n_seq) * kv->n_layers * kv->n_kv_heads;
}

tri_status check_protect(int32_t n_prompt, int32_t n_recent, int32_t budget, int32_t n_cap) {
  if (n_prompt < 0 || n_recent < 0 || budget < 1) return TRI_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_prompt) + n_recent > budget) return TRI_ERR_INVALID_ARG;
  if (budget > n_cap) return TRI_ERR_INVALID_ARG;
  return TRI_OK;
}

// 0.64 fixed-point turns per position of band f: omega_f / (2 pi).
uint64_t nu_fixed(double omega) {
  const double turns = omega / (2.0 * M_PI);  // < 0.16
  return static_cast<uint64_t>(std::ldexp(turns, 64));
}

}  // namespace
}  // namespace tri

using namespace tri;

extern "C" {

const char* tri_status_string(tri_status s) {
  switch (s) {
    case TRI_OK: return "ok";
    case TRI_ERR_INVALID_ARG: return "invalid argument";
    case TRI_ERR_UNSUPPORTED: return "unsupported head_dim, dtype or device";
    case TRI_ERR_CUDA: return "CUDA launch failed";
    case TRI_ERR_TIMEOUT: return "timed out";
  }
  return "unknown status";
}

int32_t tri_abi_version(void) { return 3; }

uint64_t tri_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

size_t tri_calibrate_workspace_bytes(int32_t n_layers, int32_t n_q_heads, int32_t group,
                                     int32_t head_dim, int64_t n_tok) {
  if (n_layers < 1 || n_q_heads < 1 || group < 1 || n_q_heads % group || head_dim < 2 || n_tok < 1)
    return 0;
  const int lh = n_layers * (n_q_heads / group);
  const int sp = calibrate_split_count(lh, static_cast<int64_t>(group) * n_tok);
  return static_cast<size_t>(lh) * sp * (head_dim / 2) * 3 * sizeof(float);
}

tri_status tri_calibrate_centers(const void* q, tri_dtype dtype, int32_t n_layers,
                                 int32_t n_q_heads, int32_t group, int32_t head_dim,
                                 int64_t n_tok, tri_rope_style style, tri_centers out,
                                 void* ws, size_t ws_bytes, tri_stream_t stream) {
  TRI_CALL_RANGE();
  if (dtype != TRI_BF16 && dtype != TRI_F32) return TRI_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return TRI_ERR_UNSUPPORTED;
  if (style != TRI_ROPE_INTERLEAVED && style != TRI_ROPE_HALF) return TRI_ERR_INVALID_ARG;
  if (!q || !aligned(q, 16) || n_layers < 1 || n_q_heads < 1 || group < 1 ||
      n_q_heads % group != 0 || n_tok < 1)
    return TRI_ERR_INVALID_ARG;
  if (!out.center || !out.mean_norm || !out.mrl || !aligned(out.center, 8) ||
      !aligned(out.mean_norm, 4) || !aligned(out.mrl, 4))
    return TRI_ERR_INVALID_ARG;
  const size_t need = tri_calibrate_workspace_bytes(n_layers, n_q_heads, group, head_dim, n_tok);
  if (ws_bytes < need || (need > 0 && (!ws || !aligned(ws, 16)))) return TRI_ERR_INVALID_ARG;
  CalibParams p{};
  p.q = q;
  p.ws = static_cast<float*>(ws);
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

namespace tri {
namespace {

// Rows per CTA of the score kernels: 32 tiles (1 MB of keys at 32 KB tiles),
// fewer for small caches; and the CTAs per slice.
void score_tiling(const tri_kv* kv, int32_t& rows_per_cta, int32_t& tiles_per_slice) {
  const ScoreGeometry g = score_geometry(kv->dtype, kv->head_dim);
  int rpc = 32 * g.tile_rows;
  const int cap_rows = (kv->n_cap + g.tile_rows - 1) / g.tile_rows * g.tile_rows;
  if (cap_rows < rpc) rpc = cap_rows;
  rows_per_cta = rpc;
  tiles_per_slice = static_cast<int32_t>((kv->n_cap + rpc - 1) / rpc);
}

// Shared by tri_score and tri_compress: argument checks and the score
// kernel's parameter block (host fp64 per-band constants).
tri_status prepare_score(const tri_kv* kv, const tri_centers* c, double rope_theta, tri_rope_style style,
                         tri_norm_mode norm_mode, const int32_t* offsets, int32_t n_offsets,
                         const int64_t* p_cur, int32_t n_prompt, int32_t n_recent, float* scores,
                         bool need_v, ScoreParams& p) {
  tri_status st = check_kv(kv, need_v);
  if (st != TRI_OK) return st;
  if (!c || !c->center || !c->mean_norm || !c->mrl || !aligned(c->center, 8)) return TRI_ERR_INVALID_ARG;
  if (style != TRI_ROPE_INTERLEAVED && style != TRI_ROPE_HALF) return TRI_ERR_INVALID_ARG;
  if (norm_mode != TRI_NORM_WEIGHTED && norm_mode != TRI_NORM_UNWEIGHTED) return TRI_ERR_INVALID_ARG;
  if (!(rope_theta > 1.0) || !std::isfinite(rope_theta)) return TRI_ERR_INVALID_ARG;
  if (!offsets || n_offsets < 1 || n_offsets > 64) return TRI_ERR_INVALID_ARG;
  if (!p_cur || !aligned(p_cur, 8) || !scores || !aligned(scores, 4)) return TRI_ERR_INVALID_ARG;
  if (n_prompt < 0 || n_recent < 0) return TRI_ERR_INVALID_ARG;

  p = ScoreParams{};
  const int D = kv->head_dim, F = D / 2;
  const ScoreGeometry g = score_geometry(kv->dtype, D);
  for (int f = 0; f < F; ++f) {
    const double omega = std::pow(rope_theta, -2.0 * f / D);
    p.nu[f] = nu_fixed(omega);
    double gr = 0.0, gi = 0.0;
    for (int j = 0; j < n_offsets; ++j) {
      gr += std::cos(omega * offsets[j]);
      gi += std::sin(omega * offsets[j]);
    }
    p.g_re[f] = static_cast<float>(gr / n_offsets);
    p.g_im[f] = static_cast<float>(gi / n_offsets);
    p.step_re[f] = static_cast<float>(std::cos(omega * g.step));
    p.step_im[f] = static_cast<float>(-std::sin(omega * g.step));
    p.jump_re[f] = static_cast<float>(std::cos(omega * g.jump));
    p.jump_im[f] = static_cast<float>(-std::sin(omega * g.jump));
  }
  p.k = kv->k;
  p.pos = kv->pos;
  p.n_valid = kv->n_valid;
  p.p_cur = p_cur;
  p.center = c->center;
  p.mean_norm = c->mean_norm;
  p.mrl = c->mrl;
  p.scores = scores;
  p.dev_status = kv->dev_status;
  p.rows = row_map(kv);
  p.n_cap = kv->n_cap;
  p.lh_count = kv->n_layers * kv->n_kv_heads;
  p.n_prompt = n_prompt;
  p.n_recent = n_recent;
  p.norm_mode = norm_mode;
  score_tiling(kv, p.rows_per_cta, p.tiles_per_slice);
  if (slices_of(kv) * p.tiles_per_slice > 0x7fffffff) return TRI_ERR_INVALID_ARG;
  return TRI_OK;
}

CompactParams compact_params(const tri_kv* kv, const int32_t* keep_idx, int32_t budget) {
  CompactParams p{};
  p.k = static_cast<char*>(kv->k);
  p.v = static_cast<char*>(kv->v);
  p.pos = kv->pos;
  p.pos_out = kv->pos_out;
  p.n_valid = kv->n_valid;
  p.keep = keep_idx;
  p.dev_status = kv->dev_status;
  p.rows = row_map(kv);
  p.n_cap = kv->n_cap;
  p.budget = budget;
  p.row_bytes = kv->head_dim * elem_bytes(kv->dtype);
  return p;
}

SelectParams select_params(const float* scores, const tri_kv* kv, int32_t n_prompt, int32_t n_recent,
                           int32_t budget, int32_t* keep_idx) {
  SelectParams p{};
  p.scores = scores;
  p.n_valid = kv->n_valid;
  p.keep = keep_idx;
  p.dev_status = kv->dev_status;
  p.n_cap = kv->n_cap;
  p.n_prompt = n_prompt;
  p.n_recent = n_recent;
  p.budget = budget;
  p.n_layers = kv->n_layers;
  p.n_kv_heads = kv->n_kv_heads;
  return p;
}

}  // namespace
}  // namespace tri

extern "C" {

tri_status tri_score(const tri_kv* kv, const tri_centers* c, double rope_theta,
                     tri_rope_style style, tri_norm_mode norm_mode, const int32_t* offsets,
                     int32_t n_offsets, const int64_t* p_cur, int32_t n_prompt,
                     int32_t n_recent, float* scores, tri_stream_t stream) {
  TRI_CALL_RANGE();
  ScoreParams p;
  const tri_status st = prepare_score(kv, c, rope_theta, style, norm_mode, offsets, n_offsets, p_cur,
                                      n_prompt, n_recent, scores, false, p);
  if (st != TRI_OK) return st;
  const cudaError_t e = launch_score(p, kv->dtype, kv->head_dim, style, pos_mode(kv),
                                     static_cast<int>(slices_of(kv)), stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

size_t tri_compress_workspace_bytes(const tri_kv* kv) {
  if (check_kv(kv, false) != TRI_OK) return 0;
  return static_cast<size_t>(slices_of(kv)) * kv->n_cap * sizeof(float);
}

tri_status tri_compress(const tri_kv* kv, const tri_centers* c, double rope_theta, tri_rope_style style,
                        tri_norm_mode norm_mode, const int32_t* offsets, int32_t n_offsets,
                        const int64_t* p_cur, int32_t n_prompt, int32_t n_recent, int32_t budget,
                        int32_t* keep_idx, void* ws, size_t ws_bytes, tri_stream_t stream) {
  TRI_CALL_RANGE();
  tri_status st = check_kv(kv, true);
  if (st != TRI_OK) return st;
  const size_t need = tri_compress_workspace_bytes(kv);
  if (need == 0 || ws_bytes < need || !ws || !aligned(ws, 16)) return TRI_ERR_INVALID_ARG;
  if (!kv->pos_out || !keep_idx || !aligned(keep_idx, 4)) return TRI_ERR_INVALID_ARG;
  ScoreParams p;
  float* scores = static_cast<float*>(ws);
  st = check_protect(n_prompt, n_recent, budget, kv->n_cap);
  if (st != TRI_OK) return st;
  st = prepare_score(kv, c, rope_theta, style, norm_mode, offsets, n_offsets, p_cur, n_prompt, n_recent,
                     scores, true, p);
  if (st != TRI_OK) return st;
  const int n_slices = static_cast<int>(slices_of(kv));
  const SelectParams ps = select_params(scores, kv, n_prompt, n_recent, budget, keep_idx);
  const CompactParams pc = compact_params(kv, keep_idx, budget);
  if (p.tiles_per_slice == 1) {
    // A slice fits one score CTA: that CTA scores, selects and compacts it
    // (one launch), so each slice's latency-bound selection overlaps other
    // slices' score and row traffic.
    const cudaError_t e = launch_compress_slices(p, ps, pc, kv->dtype, kv->head_dim, style, pos_mode(kv),
                                                 n_slices, stream);
    return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
  }
  // Several score CTAs per slice: three kernels. Selecting in the last score
  // CTA of each slice to finish measured slower: the score kernel is close to
  // its issue limit, and a selecting CTA's slot stops streaming keys.
  cudaError_t e = launch_score(p, kv->dtype, kv->head_dim, style, pos_mode(kv), n_slices, stream);
  if (e != cudaSuccess) return TRI_ERR_CUDA;
  e = launch_select(ps, n_slices, stream);
  if (e != cudaSuccess) return TRI_ERR_CUDA;
  e = launch_compact(pc, n_slices, stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

tri_status tri_select_compact(const float* scores, const tri_kv* kv, int32_t n_prompt, int32_t n_recent,
                              int32_t budget, int32_t* keep_idx, tri_stream_t stream) {
  TRI_CALL_RANGE();
  tri_status st = check_kv(kv, true);
  if (st != TRI_OK) return st;
  if (!kv->pos_out || !scores || !aligned(scores, 4) || !keep_idx || !aligned(keep_idx, 4)) return TRI_ERR_INVALID_ARG;
  st = check_protect(n_prompt, n_recent, budget, kv->n_cap);
  if (st != TRI_OK) return st;
  const cudaError_t e = launch_select_compact(select_params(scores, kv, n_prompt, n_recent, budget, keep_idx),
                                              compact_params(kv, keep_idx, budget), false,
                                              static_cast<int>(slices_of(kv)), stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

tri_status rand_evict_compact(const tri_kv* kv, uint64_t seed, uint32_t round, tri_draw_scope scope,
                              int32_t n_prompt, int32_t n_recent, int32_t budget, int32_t* keep_idx,
                              tri_stream_t stream) {
  TRI_CALL_RANGE();
  tri_status st = check_kv(kv, true);
  if (st != TRI_OK) return st;
  if (kv->n_layers > 65535 || kv->n_kv_heads > 65536) return TRI_ERR_INVALID_ARG;
  if (scope != TRI_DRAW_PER_HEAD && scope != TRI_DRAW_PER_LAYER && scope != TRI_DRAW_PER_SEQUENCE)
    return TRI_ERR_INVALID_ARG;
  if (!kv->pos_out || !keep_idx || !aligned(keep_idx, 4)) return TRI_ERR_INVALID_ARG;
  st = check_protect(n_prompt, n_recent, budget, kv->n_cap);
  if (st != TRI_OK) return st;
  SelectParams p = select_params(nullptr, kv, n_prompt, n_recent, budget, keep_idx);
  p.seed = seed;
  p.round = round;
  p.draw_scope = scope;
  const cudaError_t e = launch_select_compact(p, compact_params(kv, keep_idx, budget), true,
                                              static_cast<int>(slices_of(kv)), stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

tri_status tri_select_topk(const float* scores, const tri_kv* kv, int32_t n_prompt,
                           int32_t n_recent, int32_t budget, int32_t* keep_idx,
                           tri_stream_t stream) {
  TRI_CALL_RANGE();
  if (!kv) return TRI_ERR_INVALID_ARG;
  if (kv->n_seq < 1 || kv->n_layers < 1 || kv->n_kv_heads < 1 || kv->n_cap < 1) return TRI_ERR_INVALID_ARG;
  if (!kv->n_valid || !aligned(kv->n_valid, 4)) return TRI_ERR_INVALID_ARG;
  if (!scores || !aligned(scores, 4) || !keep_idx || !aligned(keep_idx, 4)) return TRI_ERR_INVALID_ARG;
  tri_status st = check_protect(n_prompt, n_recent, budget, kv->n_cap);
  if (st != TRI_OK) return st;
  if (slices_of(kv) > 0x7fffffff) return TRI_ERR_INVALID_ARG;
  const cudaError_t e = launch_select(select_params(scores, kv, n_prompt, n_recent, budget, keep_idx),
                                      static_cast<int>(slices_of(kv)), stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

tri_status rand_evict(const tri_kv* kv, uint64_t seed, uint32_t round, int32_t n_prompt,
                      int32_t n_recent, int32_t budget, int32_t* keep_idx, tri_stream_t stream) {
  TRI_CALL_RANGE();
  return rand_evict_scoped(kv, seed, round, TRI_DRAW_PER_HEAD, n_prompt, n_recent, budget, keep_idx, stream);
}

tri_status rand_evict_scoped(const tri_kv* kv, uint64_t seed, uint32_t round, tri_draw_scope scope,
                             int32_t n_prompt, int32_t n_recent, int32_t budget, int32_t* keep_idx,
                             tri_stream_t stream) {
  TRI_CALL_RANGE();
  if (!kv) return TRI_ERR_INVALID_ARG;
  if (scope != TRI_DRAW_PER_HEAD && scope != TRI_DRAW_PER_LAYER && scope != TRI_DRAW_PER_SEQUENCE)
    return TRI_ERR_INVALID_ARG;
  if (kv->n_seq < 1 || kv->n_layers < 1 || kv->n_kv_heads < 1 || kv->n_cap < 1) return TRI_ERR_INVALID_ARG;
  if (kv->n_layers > 65535 || kv->n_kv_heads > 65536) return TRI_ERR_INVALID_ARG;
  if (!kv->n_valid || !aligned(kv->n_valid, 4) || !keep_idx || !aligned(keep_idx, 4)) return TRI_ERR_INVALID_ARG;
  tri_status st = check_protect(n_prompt, n_recent, budget, kv->n_cap);
  if (st != TRI_OK) return st;
  if (slices_of(kv) > 0x7fffffff) return TRI_ERR_INVALID_ARG;
  SelectParams p = select_params(nullptr, kv, n_prompt, n_recent, budget, keep_idx);
  p.seed = seed;
  p.round = round;
  p.draw_scope = scope;
  const cudaError_t e = launch_rand_select(p, static_cast<int>(slices_of(kv)), stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

tri_status tri_compact_kv(const tri_kv* kv, const int32_t* keep_idx, int32_t budget,
                          tri_stream_t stream) {
  TRI_CALL_RANGE();
  tri_status st = check_kv(kv, true);
  if (st != TRI_OK) return st;
  if (!kv->pos_out) return TRI_ERR_INVALID_ARG;
  if (!keep_idx || !aligned(keep_idx, 4) || budget < 1 || budget > kv->n_cap) return TRI_ERR_INVALID_ARG;
  const cudaError_t e = launch_compact(compact_params(kv, keep_idx, budget), static_cast<int>(slices_of(kv)), stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

size_t tri_score_heads_workspace_bytes(const tri_kv* kv, int32_t group) {
  if (check_kv(kv, false) != TRI_OK || group < 1 || group > MAX_GROUP) return 0;
  int32_t rpc, tiles;
  score_tiling(kv, rpc, tiles);
  return static_cast<size_t>(slices_of(kv)) * tiles * group * 3 * sizeof(double);
}

tri_status tri_score_heads(const tri_kv* kv, const tri_centers* centers, int32_t group, double rope_theta,
                           tri_rope_style style, tri_norm_mode norm_mode, const int32_t* offsets,
                           int32_t n_offsets, const int64_t* p_cur, float* scores_g, float* stats,
                           void* ws, size_t ws_bytes, tri_stream_t stream) {
  TRI_CALL_RANGE();
  if (group < 1 || group > MAX_GROUP) return TRI_ERR_INVALID_ARG;
  if (!stats || !aligned(stats, 8)) return TRI_ERR_INVALID_ARG;
  ScoreParams p;
  tri_status st = prepare_score(kv, centers, rope_theta, style, norm_mode, offsets, n_offsets, p_cur, 0, 0,
                                scores_g, false, p);
  if (st != TRI_OK) return st;
  const size_t need = tri_score_heads_workspace_bytes(kv, group);
  if (need == 0 || ws_bytes < need || !ws || !aligned(ws, 16)) return TRI_ERR_INVALID_ARG;
  p.scores = nullptr;
  p.scores_g = scores_g;
  p.partials = static_cast<double*>(ws);
  p.group = group;
  const int n_slices = static_cast<int>(slices_of(kv));
  const bool tc = kv->dtype == TRI_BF16;
  if (tc) {
    // the tensor-core kernel's own blocks (128 rows) and runs per CTA; never
    // more CTAs per slice than the workspace query counted (its rotation
    // steps come from the fixed-point phases on the device)
    int32_t max_rpc;
    const ScoreGeometry g = tc_heads_geometry(kv->head_dim, max_rpc);
    const int32_t cap_rows = (kv->n_cap + g.tile_rows - 1) / g.tile_rows * g.tile_rows;
    p.rows_per_cta = cap_rows < max_rpc ? cap_rows : max_rpc;
    p.tiles_per_slice = (kv->n_cap + p.rows_per_cta - 1) / p.rows_per_cta;
  }
  const int per_launch = tc ? MAX_HEADS_PER_LAUNCH_TC : MAX_HEADS_PER_LAUNCH;
  for (int h0 = 0; h0 < group; h0 += per_launch) {
    p.head0 = h0;
    const int nh = group - h0 < per_launch ? group - h0 : per_launch;
    const cudaError_t e = tc ? launch_score_heads_tc(p, nh, kv->head_dim, style, pos_mode(kv), n_slices, stream)
                             : launch_score_heads(p, nh, kv->dtype, kv->head_dim, style, pos_mode(kv),
                                                  n_slices, stream);
    if (e != cudaSuccess) return TRI_ERR_CUDA;
  }
  const cudaError_t e = launch_heads_stats(p.partials, stats, n_slices, p.tiles_per_slice, group, stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

tri_status tri_select_topk_zmax(const float* scores_g, const float* stats, int32_t group, const tri_kv* kv,
                                int32_t n_prompt, int32_t n_recent, int32_t budget, int32_t* keep_idx,
                                float* final_scores, tri_stream_t stream) {
  TRI_CALL_RANGE();
  if (!kv) return TRI_ERR_INVALID_ARG;
  if (kv->n_seq < 1 || kv->n_layers < 1 || kv->n_kv_heads < 1 || kv->n_cap < 1) return TRI_ERR_INVALID_ARG;
  if (!kv->n_valid || !aligned(kv->n_valid, 4)) return TRI_ERR_INVALID_ARG;
  if (group < 1 || group > MAX_GROUP) return TRI_ERR_INVALID_ARG;
  if (!scores_g || !aligned(scores_g, 4) || !stats || !aligned(stats, 8)) return TRI_ERR_INVALID_ARG;
  if (!keep_idx || !aligned(keep_idx, 4)) return TRI_ERR_INVALID_ARG;
  if (final_scores && !aligned(final_scores, 4)) return TRI_ERR_INVALID_ARG;
  tri_status st = check_protect(n_prompt, n_recent, budget, kv->n_cap);
  if (st != TRI_OK) return st;
  if (slices_of(kv) > 0x7fffffff) return TRI_ERR_INVALID_ARG;
  const int n_slices = static_cast<int>(slices_of(kv));
  if (final_scores) {
    const cudaError_t e = launch_zmax_scores(scores_g, stats, kv->n_valid, 1, final_scores, n_slices, kv->n_cap,
                                             group, stream);
    if (e != cudaSuccess) return TRI_ERR_CUDA;
  }
  SelectParams p = select_params(scores_g, kv, n_prompt, n_recent, budget, keep_idx);
  p.stats = stats;
  p.group = group;
  const cudaError_t e = launch_select_zmax(p, n_slices, stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

namespace {
// Workspace of tri_select_union: the heads' own picks [S][bk] int32, then
// stats [S][2] f32, the union bitmaps [groups][words] u32, the member counts
// [groups] int32 (each part 16-byte aligned).
struct UnionWs {
  int32_t bk;
  int32_t words;
  size_t keepk_off, stats_off, member_off, count_off, total;
};
size_t align16(size_t x) { return (x + 15) / 16 * 16; }
UnionWs union_ws(const tri_kv* kv, int32_t n_prompt, int32_t n_recent, int32_t k_head) {
  UnionWs u{};
  const int64_t S = slices_of(kv);
  const int64_t groups = S / kv->n_kv_heads;
  const int64_t bk = (k_head <= 0) ? 0 : std::min<int64_t>(static_cast<int64_t>(n_prompt) + n_recent + k_head,
                                                           kv->n_cap);
  u.bk = static_cast<int32_t>(bk);
  u.words = (kv->n_cap + 31) / 32;
  u.keepk_off = 0;
  u.stats_off = align16(u.keepk_off + static_cast<size_t>(S) * bk * sizeof(int32_t));
  u.member_off = align16(u.stats_off + static_cast<size_t>(S) * 2 * sizeof(float));
  u.count_off = align16(u.member_off + static_cast<size_t>(groups) * u.words * sizeof(uint32_t));
  u.total = align16(u.count_off + static_cast<size_t>(groups) * sizeof(int32_t));
  return u;
}
constexpr int32_t UNION_MAX_CAP = 524288;
}  // namespace

size_t tri_select_union_workspace_bytes(const tri_kv* kv, int32_t n_prompt, int32_t n_recent, int32_t k_head) {
  if (!kv || kv->n_seq < 1 || kv->n_layers < 1 || kv->n_kv_heads < 1 || kv->n_cap < 1) return 0;
  if (n_prompt < 0 || n_recent < 0 || k_head < 0) return 0;
  return union_ws(kv, n_prompt, n_recent, k_head).total;
}

tri_status tri_select_union(const float* scores, const tri_kv* kv, int32_t n_prompt, int32_t n_recent,
                            int32_t budget, int32_t k_head, int32_t* keep_idx, float* final_scores, void* ws,
                            size_t ws_bytes, tri_stream_t stream) {
  TRI_CALL_RANGE();
  if (!kv) return TRI_ERR_INVALID_ARG;
  if (kv->n_seq < 1 || kv->n_layers < 1 || kv->n_kv_heads < 1 || kv->n_cap < 1) return TRI_ERR_INVALID_ARG;
  if (kv->n_kv_heads > MAX_GROUP || kv->n_cap > UNION_MAX_CAP) return TRI_ERR_UNSUPPORTED;
  if (!kv->n_valid || !aligned(kv->n_valid, 4)) return TRI_ERR_INVALID_ARG;
  if (!scores || !aligned(scores, 4) || !keep_idx || !aligned(keep_idx, 4) || k_head < 0) return TRI_ERR_INVALID_ARG;
  if (final_scores && !aligned(final_scores, 4)) return TRI_ERR_INVALID_ARG;
  tri_status st = check_protect(n_prompt, n_recent, budget, kv->n_cap);
  if (st != TRI_OK) return st;
  if (slices_of(kv) > 0x7fffffff) return TRI_ERR_INVALID_ARG;
  const UnionWs u = union_ws(kv, n_prompt, n_recent, k_head);
  if (!ws || !aligned(ws, 16) || ws_bytes < u.total) return TRI_ERR_INVALID_ARG;
  const int n_slices = static_cast<int>(slices_of(kv));
  const int n_groups = n_slices / kv->n_kv_heads;
  char* base = static_cast<char*>(ws);
  int32_t* keepk = reinterpret_cast<int32_t*>(base + u.keepk_off);
  float* stats = reinterpret_cast<float*>(base + u.stats_off);
  uint32_t* member = reinterpret_cast<uint32_t*>(base + u.member_off);
  int32_t* ucount = reinterpret_cast<int32_t*>(base + u.count_off);
  cudaError_t e;
  if (u.bk > 0) {  // 1. every head's own picks
    e = launch_select(select_params(scores, kv, n_prompt, n_recent, u.bk, keepk), n_slices, stream);
    if (e != cudaSuccess) return TRI_ERR_CUDA;
  }
  e = launch_slice_stats(scores, kv->n_valid, stats, n_slices, kv->n_cap, stream);  // 2. statistics
  if (e != cudaSuccess) return TRI_ERR_CUDA;
  UnionPrepParams q{};  // 3. the union
  q.scores = scores;
  q.n_valid = kv->n_valid;
  q.keepk = keepk;
  q.member = member;
  q.ucount = ucount;
  q.dev_status = kv->dev_status;
  q.n_cap = kv->n_cap;
  q.bk = u.bk;
  q.n_prompt = n_prompt;
  q.n_recent = n_recent;
  q.group = kv->n_kv_heads;
  q.member_words = u.words;
  e = launch_union_prep(q, n_groups, stream);
  if (e != cudaSuccess) return TRI_ERR_CUDA;
  if (final_scores) {
    e = launch_zmax_scores(scores, stats, kv->n_valid, kv->n_kv_heads, final_scores, n_groups, kv->n_cap,
                           kv->n_kv_heads, stream);
    if (e != cudaSuccess) return TRI_ERR_CUDA;
  }
  SelectParams p = select_params(scores, kv, n_prompt, n_recent, budget, keep_idx);  // 4. one list per group
  p.stats = stats;
  p.group = kv->n_kv_heads;
  p.member = member;
  p.ucount = ucount;
  p.member_words = u.words;
  e = launch_select_union(p, n_groups, stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

tri_status tri_paged_blocks_used(const tri_kv* kv, int32_t* blocks_used, tri_stream_t stream) {
  TRI_CALL_RANGE();
  tri_status st = check_kv(kv, false);
  if (st != TRI_OK) return st;
  if (!kv->block_table || !blocks_used || !aligned(blocks_used, 4)) return TRI_ERR_INVALID_ARG;
  const cudaError_t e = launch_blocks_used(row_map(kv), kv->n_valid, blocks_used, kv->n_seq, stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

tri_status tri_selftest_wait_timeout(int32_t* dev_status, uint64_t limit_ns, tri_stream_t stream) {
  TRI_CALL_RANGE();
  if (!dev_status || !aligned(dev_status, 4) || limit_ns < 1000u || limit_ns > 1000000000u) return TRI_ERR_INVALID_ARG;
  const cudaError_t e = launch_wait_timeout_selftest(dev_status, limit_ns, stream);
  return e == cudaSuccess ? TRI_OK : TRI_ERR_CUDA;
}

}  // extern "C"
