// tri_oracle.cpp -- the ORACLE for the KV-cache compression hot path.
//
// TEST INFRASTRUCTURE ONLY. This file is a plain, slow, obviously correct CPU
// restatement of what the hot path computes, in fp64, one slice (one sequence,
// layer and KV head) at a time. Only the tests, the smoke check and the bench's
// CPU-baseline leg may load it. The product path (the CUDA library) shares no
// code, header, table or constant with it and never calls it.
//
// Sources, by page title and section / equation:
//   [TA]  "TriAttention: Efficient Long Reasoning with Trigonometric KV
//         Compression" (paper summary page), section 3.4, sub-sections
//         "Mathematical Foundation: RoPE Attention as a Trigonometric Series",
//         "TriAttention Key Importance Scoring: The Trigonometric Series Term",
//         "... The Norm-Based Term", "Adaptive Weighting via Q/K Concentration",
//         "Handling Multiple Future Positions", "KV Cache Pruning Procedure",
//         "Offline Calibration Procedure".
//   [TB]  the TriAttention blog page (same title), sections "TriAttention
//         Scoring" and the S_norm part (extra_coef = E|q_f| - |E q_f|).
//   [RA]  "Random Attention: Rethinking KV Cache Eviction for Efficient
//         Reasoning", section 2 (Eq. 2, periodic eviction with budget K and
//         buffer r), section 3 (Eq. 3, Algorithm 1), Appendix F (keep-sets
//         sorted chronologically, then compacted with a gather).
//   [PX]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
//         1, 2, 3" (SC'11): the Philox-4x32 round and its Weyl key schedule.
//
// Readings where the pages leave a step open (each one is listed with its
// reason in the design notes of the repository):
//   * keys are stored pre-RoPE, with a position per row (slot index when no
//     position array is given);
//   * the G query heads of a GQA group are pooled into one centre per KV head
//     (orc_zscore_max implements the paper's per-query-head alternative);
//   * p_cur, the position of the newest cached token, is the "current query
//     position"; a key's age is p_cur - p_i;
//   * budget B counts every survivor, protected rows included;
//   * equal scores keep the lower slot index; NaN ranks below everything.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -shared -fPIC (see oracle/__init__.py).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

// [TA] "RoPE in complex form": band f rotates at omega_f = theta^(-2f/d).
double band_omega(int64_t f, int64_t d, double theta) {
  return std::pow(theta, -2.0 * static_cast<double>(f) / static_cast<double>(d));
}

// The complex value of band f of a real d-vector. style 0 pairs
// (x_{2f}, x_{2f+1}) as [TA] writes it; style 1 pairs (x_f, x_{f+d/2}), the
// "half" rotation style the blog's invert_rope call names.
void band_of(const double* x, int64_t f, int64_t d, int style, double* re, double* im) {
  if (style == 0) {
    *re = x[2 * f];
    *im = x[2 * f + 1];
  } else {
    *re = x[f];
    *im = x[f + d / 2];
  }
}

void set_band(double* x, int64_t f, int64_t d, int style, double re, double im) {
  if (style == 0) {
    x[2 * f] = re;
    x[2 * f + 1] = im;
  } else {
    x[f] = re;
    x[f + d / 2] = im;
  }
}

// Explicit RoPE: rotate every band of x by omega_f * p ([TA] "RoPE in complex
// form": multiply x_f by e^{i omega_f p}), written as a 2x2 rotation.
void rope_rotate(const double* x, int64_t d, int style, double theta, double p, double* out) {
  const int64_t F = d / 2;
  for (int64_t f = 0; f < F; ++f) {
    double a, b;
    band_of(x, f, d, style, &a, &b);
    const double ang = band_omega(f, d, theta) * p;
    const double c = std::cos(ang), s = std::sin(ang);
    set_band(out, f, d, style, a * c - b * s, a * s + b * c);
  }
}

// Norm weight of band f: (1 - R_f) E|q_f| for the weighted S_norm of [TA]
// "Adaptive Weighting via Q/K Concentration"; E|q_f| alone for the unweighted
// S_norm^(0) of [TA] "The Norm-Based Term" (norm_mode 1).
double norm_weight(const double* mean_norm, const double* mrl, int64_t f, int norm_mode) {
  if (norm_mode == 1) return mean_norm[f];
  return (1.0 - mrl[f]) * mean_norm[f];
}

}  // namespace

extern "C" {

int orc_abi_version() { return 1; }

// ---------------------------------------------------------------------------
// Offline calibration, [TA] "Offline Calibration Procedure": per head and band,
// the centre E[q_f] (a complex mean), the mean magnitude E|q_f| and the Mean
// Resultant Length R_f = |E q_f| / E|q_f| ([TA] "Measurement via Mean
// Resultant Length"). The G query heads that share KV head h (query heads
// h*G .. h*G+G-1) are pooled into one sample set.
//
// q: [L][Hq][n_tok][d] pre-RoPE queries. Outputs per (layer*Hkv + h):
// center [.][F][2] (re, im), mean_norm [.][F], mrl [.][F]. When every sample
// of a band is zero, R is taken as 0.
// ---------------------------------------------------------------------------
void orc_calibrate(const double* q, int64_t L, int64_t Hq, int64_t G, int64_t n_tok, int64_t d,
                   int style, double* center, double* mean_norm, double* mrl) {
  const int64_t Hkv = Hq / G, F = d / 2;
  for (int64_t l = 0; l < L; ++l)
    for (int64_t h = 0; h < Hkv; ++h)
      for (int64_t f = 0; f < F; ++f) {
        double sum_re = 0.0, sum_im = 0.0, sum_abs = 0.0;
        for (int64_t g = 0; g < G; ++g) {
          const int64_t qh = h * G + g;
          for (int64_t t = 0; t < n_tok; ++t) {
            const double* x = q + ((l * Hq + qh) * n_tok + t) * d;
            double re, im;
            band_of(x, f, d, style, &re, &im);
            sum_re += re;
            sum_im += im;
            sum_abs += std::hypot(re, im);
          }
        }
        const double n = static_cast<double>(G * n_tok);
        const double c_re = sum_re / n, c_im = sum_im / n, m = sum_abs / n;
        const int64_t o = (l * Hkv + h) * F + f;
        center[2 * o] = c_re;
        center[2 * o + 1] = c_im;
        mean_norm[o] = m;
        mrl[o] = (m > 0.0) ? std::hypot(c_re, c_im) / m : 0.0;
      }
}

// ---------------------------------------------------------------------------
// Score by the direct series, one slice.
//   S_trig(k, Delta) = sum_f |E q_f| |k_f| cos(omega_f Delta + phi_f),
//       phi_f = arg E[q_f] - arg k_f           ([TA] "The Trigonometric Series Term")
//   S_norm(k)        = sum_f (1 - R_f) E|q_f| |k_f|   ([TA] "Adaptive Weighting ...")
//   S(k, Delta)      = S_trig + S_norm          ([TA] "The combined score")
//   S~(k) = (1/|D|) sum_{delta in D} S(k, age + delta), age = p_cur - p_k
//                                               ([TA] "Handling Multiple Future Positions")
// k: [n][d] pre-RoPE keys; pos: [n] positions or NULL (slot index); center
// [F][2], mean_norm [F], mrl [F] of this slice's KV head. norm_mode 0 =
// weighted S_norm, 1 = unweighted S_norm^(0). out: [n]. *cos_count (if not
// NULL) is increased by the number of cosines evaluated ([TA] counts
// B x |D| x d/2 of them per pruning step).
// ---------------------------------------------------------------------------
void orc_score_series(const double* k, const int64_t* pos, int64_t n, int64_t d, int style,
                      double theta, const double* center, const double* mean_norm,
                      const double* mrl, const int64_t* offsets, int64_t n_off, int64_t p_cur,
                      int norm_mode, double* out, int64_t* cos_count) {
  const int64_t F = d / 2;
  std::vector<double> omega(F), c_abs(F), c_arg(F);
  for (int64_t f = 0; f < F; ++f) {
    omega[f] = band_omega(f, d, theta);
    c_abs[f] = std::hypot(center[2 * f], center[2 * f + 1]);
    c_arg[f] = std::atan2(center[2 * f + 1], center[2 * f]);
  }
  int64_t cosines = 0;
  for (int64_t i = 0; i < n; ++i) {
    const double* key = k + i * d;
    const int64_t p = pos ? pos[i] : i;
    const double age = static_cast<double>(p_cur - p);
    double s_norm = 0.0, s_trig_sum = 0.0;
    for (int64_t f = 0; f < F; ++f) {
      double kr, ki;
      band_of(key, f, d, style, &kr, &ki);
      const double k_abs = std::hypot(kr, ki);
      const double phi = c_arg[f] - std::atan2(ki, kr);
      for (int64_t j = 0; j < n_off; ++j) {
        const double delta = age + static_cast<double>(offsets[j]);
        s_trig_sum += c_abs[f] * k_abs * std::cos(omega[f] * delta + phi);
        ++cosines;
      }
      s_norm += norm_weight(mean_norm, mrl, f, norm_mode) * k_abs;
    }
    // S_norm does not depend on Delta, so its average over D is itself.
    out[i] = s_trig_sum / static_cast<double>(n_off) + s_norm;
  }
  if (cos_count) *cos_count += cosines;
}

// ---------------------------------------------------------------------------
// RoPE of whole rows ([TA] "RoPE in complex form"; [TB] "scoring": an engine
// stores post-RoPE keys and invert_rope undoes the rotation before scoring):
// row i of x is rotated by +omega_f pos_i (sign = +1, what an engine stores)
// or by -omega_f pos_i (sign = -1, the inverse). x, out: [n][d]; pos [n].
// ---------------------------------------------------------------------------
void orc_rope_rows(const double* x, const int64_t* pos, int64_t n, int64_t d, int style, double theta,
                   int sign, double* out) {
  for (int64_t i = 0; i < n; ++i)
    rope_rotate(x + i * d, d, style, theta, static_cast<double>(sign) * static_cast<double>(pos[i]),
                out + i * d);
}

// ---------------------------------------------------------------------------
// Score by brute force, one slice (tiny inputs only). The centre, written as a
// real d-vector, stands in for a future query ([TA] "Why the Q center, not
// actual queries"): rotate it to p_cur + delta and the key to p_k with
// explicit RoPE rotations, take the real dot product (the attention logit of
// [TA] "The attention dot product in complex form"), average over D, and add
// the same norm term. It must equal orc_score_series to rounding.
// ---------------------------------------------------------------------------
void orc_score_bruteforce(const double* k, const int64_t* pos, int64_t n, int64_t d, int style,
                          double theta, const double* center, const double* mean_norm,
                          const double* mrl, const int64_t* offsets, int64_t n_off,
                          int64_t p_cur, int norm_mode, double* out) {
  const int64_t F = d / 2;
  std::vector<double> cvec(d), cq(d), kk(d);
  for (int64_t f = 0; f < F; ++f) set_band(cvec.data(), f, d, style, center[2 * f], center[2 * f + 1]);
  for (int64_t i = 0; i < n; ++i) {
    const double* key = k + i * d;
    const int64_t p = pos ? pos[i] : i;
    rope_rotate(key, d, style, theta, static_cast<double>(p), kk.data());
    double logit_sum = 0.0;
    for (int64_t j = 0; j < n_off; ++j) {
      rope_rotate(cvec.data(), d, style, theta, static_cast<double>(p_cur + offsets[j]), cq.data());
      double dot = 0.0;
      for (int64_t e = 0; e < d; ++e) dot += cq[e] * kk[e];
      logit_sum += dot;
    }
    double s_norm = 0.0;
    for (int64_t f = 0; f < F; ++f) {
      double kr, ki;
      band_of(key, f, d, style, &kr, &ki);
      s_norm += norm_weight(mean_norm, mrl, f, norm_mode) * std::hypot(kr, ki);
    }
    out[i] = logit_sum / static_cast<double>(n_off) + s_norm;
  }
}

// ---------------------------------------------------------------------------
// Budgeted selection, one slice: keep the protected prompt [0, P) and recent
// window [n_valid - W, n_valid), and the top (B - P - W) candidates of
// [P, n_valid - W) by score ([TA] "Retention and eviction": top-B by final
// score; [RA] Eq. 2 with the prompt forced in by Eq. 3 and the never-scored
// buffer of section 2). Ties keep the lower slot index; NaN ranks lowest.
// The keep list is written in ascending (chronological) order ([RA] Appendix F).
// When n_valid <= B nothing is evicted: keep = 0..n_valid-1, then -1 padding.
// keep: [B]. Returns 0, or -1 when B < P + W and eviction is needed.
// ---------------------------------------------------------------------------
int orc_select(const double* score, int64_t n_valid, int64_t P, int64_t W, int64_t B,
               int32_t* keep) {
  if (n_valid <= B) {
    for (int64_t j = 0; j < B; ++j) keep[j] = (j < n_valid) ? static_cast<int32_t>(j) : -1;
    return 0;
  }
  if (B < P + W) return -1;
  std::vector<int64_t> cand;
  for (int64_t i = P; i < n_valid - W; ++i) cand.push_back(i);
  auto better = [&](int64_t a, int64_t b) {
    const bool na = std::isnan(score[a]), nb = std::isnan(score[b]);
    if (na || nb) return !na && nb;
    return score[a] > score[b];
  };
  std::stable_sort(cand.begin(), cand.end(), better);
  std::vector<int64_t> kept;
  for (int64_t i = 0; i < P; ++i) kept.push_back(i);
  for (int64_t j = 0; j < B - P - W; ++j) kept.push_back(cand[j]);
  for (int64_t i = n_valid - W; i < n_valid; ++i) kept.push_back(i);
  std::sort(kept.begin(), kept.end());
  for (int64_t j = 0; j < B; ++j) keep[j] = static_cast<int32_t>(kept[j]);
  return 0;
}

// ---------------------------------------------------------------------------
// In-place compaction, one slice: for j ascending, row j <- row keep[j]
// ([RA] Appendix F: keep-sets sorted chronologically, KV tensors compacted
// with a gather). rows: [n_rows][row_bytes]; keep as written by orc_select
// (ascending, -1 padding ends the list). Returns the number of kept rows.
// ---------------------------------------------------------------------------
int64_t orc_compact(uint8_t* rows, int64_t row_bytes, const int32_t* keep, int64_t B) {
  int64_t j = 0;
  for (; j < B; ++j) {
    if (keep[j] < 0) break;
    if (keep[j] != j) std::memcpy(rows + j * row_bytes, rows + static_cast<int64_t>(keep[j]) * row_bytes, row_bytes);
  }
  return j;
}

// ---------------------------------------------------------------------------
// Philox-4x32 with 10 rounds [PX]. One round maps (x0, x1, x2, x3) with key
// (k0, k1) to
//   ( hi(M1*x2) ^ x1 ^ k0,  lo(M1*x2),  hi(M0*x0) ^ x3 ^ k1,  lo(M0*x0) ),
// M0 = 0xD2511F53, M1 = 0xCD9E8D57; between rounds the key is bumped by the
// Weyl constants (0x9E3779B9, 0xBB67AE85).
// ---------------------------------------------------------------------------
void orc_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * x0;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * x2;
    const uint32_t y0 = static_cast<uint32_t>(p1 >> 32) ^ x1 ^ k0;
    const uint32_t y1 = static_cast<uint32_t>(p1);
    const uint32_t y2 = static_cast<uint32_t>(p0 >> 32) ^ x3 ^ k1;
    const uint32_t y3 = static_cast<uint32_t>(p0);
    x0 = y0;
    x1 = y1;
    x2 = y2;
    x3 = y3;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

// The uniform draw u_i of [RA] Eq. 3 for slot i of one slice, as a 32-bit
// integer (u_i / 2^32 is the Uniform(0,1) value; comparing the integers
// compares the draws). Counter = (i / 4, head + 65536 * layer, seq, round),
// key = (low, high) 32 bits of the seed; word i % 4 of the output.
uint32_t orc_rand_u32(uint64_t seed, uint32_t round, int64_t seq, int64_t layer, int64_t head,
                      int64_t i) {
  const uint32_t ctr[4] = {static_cast<uint32_t>(i >> 2),
                           static_cast<uint32_t>(head + 65536 * layer),
                           static_cast<uint32_t>(seq), round};
  const uint32_t key[2] = {static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return out[i & 3];
}

// ---------------------------------------------------------------------------
// Random Attention selection, one slice ([RA] section 3, Eq. 3 and
// Algorithm 1): the prompt [0, P) scores +inf (always kept), the recent buffer
// [n_valid - W, n_valid) is never scored and kept ([RA] section 2), and every
// other slot draws u_i; keep the top (B - P - W) by (u desc, slot asc). Output
// as orc_select. Returns 0, or -1 when B < P + W and eviction is needed.
// ---------------------------------------------------------------------------
int orc_rand_select(uint64_t seed, uint32_t round, int64_t seq, int64_t layer, int64_t head,
                    int64_t n_valid, int64_t P, int64_t W, int64_t B, int32_t* keep) {
  if (n_valid <= B) {
    for (int64_t j = 0; j < B; ++j) keep[j] = (j < n_valid) ? static_cast<int32_t>(j) : -1;
    return 0;
  }
  if (B < P + W) return -1;
  std::vector<std::pair<uint32_t, int64_t>> cand;
  for (int64_t i = P; i < n_valid - W; ++i)
    cand.emplace_back(orc_rand_u32(seed, round, seq, layer, head, i), i);
  std::sort(cand.begin(), cand.end(), [](const std::pair<uint32_t, int64_t>& a,
                                         const std::pair<uint32_t, int64_t>& b) {
    if (a.first != b.first) return a.first > b.first;
    return a.second < b.second;
  });
  std::vector<int64_t> kept;
  for (int64_t i = 0; i < P; ++i) kept.push_back(i);
  for (int64_t j = 0; j < B - P - W; ++j) kept.push_back(cand[j].second);
  for (int64_t i = n_valid - W; i < n_valid; ++i) kept.push_back(i);
  std::sort(kept.begin(), kept.end());
  for (int64_t j = 0; j < B; ++j) keep[j] = static_cast<int32_t>(kept[j]);
  return 0;
}

// ---------------------------------------------------------------------------
// GQA aggregation, [TA] "Handling Grouped-Query Attention (GQA)": each of the
// G query heads that share a KV head scores every cached key with its own
// centre statistics; head g's scores are standardised with their own mean
// mu_g and standard deviation sigma_g (taken over the n keys in the cache), and
// the final score of a key is the largest z-score over the G heads.
// Readings: sigma_g is the population standard deviation (sum over n, divided
// by n); the choice scales every head of a slice alike, so no selection can
// depend on it. A head whose scores are all equal (sigma_g = 0) gives every
// key a z-score of 0.
// scores: [G][n] (head-major). Outputs mean[G], stdev[G], final_score[n].
// ---------------------------------------------------------------------------
void orc_zscore_max(const double* scores, int64_t G, int64_t n, double* mean, double* stdev,
                    double* final_score) {
  for (int64_t g = 0; g < G; ++g) {
    const double* s = scores + g * n;
    double sum = 0.0;
    for (int64_t i = 0; i < n; ++i) sum += s[i];
    const double mu = (n > 0) ? sum / static_cast<double>(n) : 0.0;
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) ss += (s[i] - mu) * (s[i] - mu);
    mean[g] = mu;
    stdev[g] = (n > 0) ? std::sqrt(ss / static_cast<double>(n)) : 0.0;
  }
  for (int64_t i = 0; i < n; ++i) {
    double best = -std::numeric_limits<double>::infinity();
    for (int64_t g = 0; g < G; ++g) {
      const double z = (stdev[g] > 0.0) ? (scores[g * n + i] - mean[g]) / stdev[g] : 0.0;
      if (z > best) best = z;
    }
    final_score[i] = best;
  }
}

// ---------------------------------------------------------------------------
// Union-based selection across heads ([TB] "eviction (union-based
// selection)"): the H heads that must share one keep-set (here the KV heads
// of one (seq, layer)) each pick their own top candidates; the union of those
// picks is kept first, ranked by a combined score, and if it holds fewer than
// the budget the rest is filled by the combined score.
// Readings: each head picks its top k_head candidates (score desc, slot asc,
// NaN lowest); the combined score is [TA]'s normalise-then-max (per-head
// z-score over all n rows, population std, then the maximum over heads, as
// orc_zscore_max); the final order is (in the union first, combined score
// desc, slot asc); prompt [0, P) and recent [n - W, n) are kept as in
// orc_select. scores: [H][n]. member: [n] out (1 = in the union), combined:
// [n] out, keep: [B] out. Returns 0, or -1 when B < P + W and eviction is
// needed.
// ---------------------------------------------------------------------------
namespace {
bool ranks_higher(double a, double b) {  // a above b; NaN lowest
  if (std::isnan(a)) return false;
  if (std::isnan(b)) return true;
  return a > b;
}
}  // namespace

// Step 1: the union of every head's top k_head candidates [P, n - W) by its
// own score (score desc, slot asc, NaN lowest). member: [n] out.
void orc_union_members(const double* scores, int64_t H, int64_t n, int64_t P, int64_t W, int64_t k_head,
                       int32_t* member) {
  for (int64_t i = 0; i < n; ++i) member[i] = 0;
  std::vector<int64_t> cand;
  for (int64_t i = P; i < n - W; ++i) cand.push_back(i);
  for (int64_t h = 0; h < H; ++h) {
    const double* s = scores + h * n;
    std::vector<int64_t> order = cand;
    std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) { return ranks_higher(s[a], s[b]); });
    const int64_t take = std::min<int64_t>(k_head, static_cast<int64_t>(order.size()));
    for (int64_t j = 0; j < take; ++j) member[order[j]] = 1;
  }
}

// Step 2: keep [0, P), then B - P - W candidates in the order (member first,
// combined desc with NaN lowest, slot asc), then [n - W, n); ascending.
// Returns 0, or -1 when B < P + W and eviction is needed.
int orc_union_rank(const int32_t* member, const double* combined, int64_t n, int64_t P, int64_t W, int64_t B,
                   int32_t* keep) {
  if (n <= B) {
    for (int64_t j = 0; j < B; ++j) keep[j] = (j < n) ? static_cast<int32_t>(j) : -1;
    return 0;
  }
  if (B < P + W) return -1;
  std::vector<int64_t> order;
  for (int64_t i = P; i < n - W; ++i) order.push_back(i);
  std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
    if (member[a] != member[b]) return member[a] > member[b];
    return ranks_higher(combined[a], combined[b]);
  });
  std::vector<int64_t> kept;
  for (int64_t i = 0; i < P; ++i) kept.push_back(i);
  for (int64_t j = 0; j < B - P - W; ++j) kept.push_back(order[j]);
  for (int64_t i = n - W; i < n; ++i) kept.push_back(i);
  std::sort(kept.begin(), kept.end());
  for (int64_t j = 0; j < B; ++j) keep[j] = static_cast<int32_t>(kept[j]);
  return 0;
}

// Both steps, with the combined score of orc_zscore_max.
int orc_union_select(const double* scores, int64_t H, int64_t n, int64_t P, int64_t W, int64_t B,
                     int64_t k_head, int32_t* member, double* combined, int32_t* keep) {
  std::vector<double> mean(H), stdev(H);
  orc_zscore_max(scores, H, n, mean.data(), stdev.data(), combined);
  if (n <= B) {
    for (int64_t i = 0; i < n; ++i) member[i] = 0;
  } else {
    orc_union_members(scores, H, n, P, W, k_head, member);
  }
  return orc_union_rank(member, combined, n, P, W, B, keep);
}

}  // extern "C"
