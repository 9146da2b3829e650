"""The oracle: a plain fp64 CPU restatement of the KV-cache compression path.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. The
product path (the CUDA library under ``kv_cache_compression_tri_gb300``)
shares no code with it and never calls it.

The arithmetic lives in ``tri_oracle.cpp`` (C++17, fp64); this module only
builds it with g++ when the shared object is missing or older than its
source, and marshals numpy arrays through ctypes. Each wrapper names the
passage it follows in the C++ file.

Parity status of each function (what pins it, all in ``tests/test_oracle_*``):
  calibrate          -- closed forms (identical samples: R = 1; symmetric
                        samples: c = 0, R = 0), the blog's three-vector MRL
                        example, the (1-R)m = m - |c| identity.
  score_series       -- brute-force RoPE rotation + dot product (exact
                        identity), hand-entered omega values, closed-form
                        single-band cases, the cosine count of the pages.
  score_bruteforce   -- the explicit RoPE definition itself; pinned by the
                        hand-entered rotation cases.
  select             -- full sort by (score desc, index asc) in Python,
                        invariants, weighted-norm top-k special case.
  compact            -- out-of-place numpy gather from a pristine copy.
  philox4x32_10      -- Triton's Philox (run by its CPU interpreter) and
                        uniformity statistics.
  rand_select        -- inclusion frequency, the survival-by-age law of
                        Random Attention, slot coverage across heads.
  rope_rows          -- the rotation itself: a round trip is the identity,
                        one band is the complex product by e^{i w p}.
  score_post_rope    -- inverse RoPE, then score_series; equals the
                        pre-RoPE score of the un-rotated keys.
  score_heads        -- per-query-head scores: score_series once per head;
                        identical heads reduce to the pooled score.
  union_select       -- brute-force set construction on tiny inputs; with
                        k_head >= the number kept it reduces to the top by
                        the z-score maximum, with k_head = 0 likewise; a
                        single head gives the plain selection.
  zscore_max         -- a hand-worked two-head example in closed form,
                        invariance under a positive affine map of any head,
                        unit variance of every z-scored head, constant heads.
  score_bound        -- hand-entered values for both band pairings;
                        |score_series| <= M (weighted norm term) and
                        0 <= score <= 2M (unweighted) on calibrated random
                        cases; equality for a zero query centre and for an
                        aligned concentrated band (tests/test_oracle_bound.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tri_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libtri_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-shared", "-fPIC", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, i32, u32, u64, dbl = (ctypes.c_int64, ctypes.c_int, ctypes.c_uint32,
                                       ctypes.c_uint64, ctypes.c_double)
            vp = ctypes.c_void_p
            lib.orc_abi_version.restype = i32
            lib.orc_calibrate.argtypes = [vp, i64, i64, i64, i64, i64, i32, vp, vp, vp]
            lib.orc_calibrate.restype = None
            lib.orc_score_series.argtypes = [vp, vp, i64, i64, i32, dbl, vp, vp, vp, vp, i64, i64,
                                             i32, vp, vp]
            lib.orc_score_series.restype = None
            lib.orc_score_bruteforce.argtypes = [vp, vp, i64, i64, i32, dbl, vp, vp, vp, vp, i64,
                                                 i64, i32, vp]
            lib.orc_score_bruteforce.restype = None
            lib.orc_select.argtypes = [vp, i64, i64, i64, i64, vp]
            lib.orc_select.restype = i32
            lib.orc_compact.argtypes = [vp, i64, vp, i64]
            lib.orc_compact.restype = i64
            lib.orc_philox4x32_10.argtypes = [vp, vp, vp]
            lib.orc_philox4x32_10.restype = None
            lib.orc_rand_u32.argtypes = [u64, u32, i64, i64, i64, i64]
            lib.orc_rand_u32.restype = u32
            lib.orc_rand_select.argtypes = [u64, u32, i64, i64, i64, i64, i64, i64, i64, vp]
            lib.orc_rand_select.restype = i32
            lib.orc_rope_rows.argtypes = [vp, vp, i64, i64, i32, dbl, i32, vp]
            lib.orc_rope_rows.restype = None
            lib.orc_union_select.argtypes = [vp, i64, i64, i64, i64, i64, i64, vp, vp, vp]
            lib.orc_union_select.restype = i32
            lib.orc_union_members.argtypes = [vp, i64, i64, i64, i64, i64, vp]
            lib.orc_union_members.restype = None
            lib.orc_union_rank.argtypes = [vp, vp, i64, i64, i64, i64, vp]
            lib.orc_union_rank.restype = i32
            lib.orc_zscore_max.argtypes = [vp, i64, i64, vp, vp, vp]
            lib.orc_zscore_max.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


ROPE_INTERLEAVED = 0
ROPE_HALF = 1
NORM_WEIGHTED = 0
NORM_UNWEIGHTED = 1


def calibrate(q, group: int, style: int = ROPE_INTERLEAVED):
    """Per-KV-head centre, mean norm and MRL from pre-RoPE queries q [L][Hq][n][d].

    TriAttention summary page, "Offline Calibration Procedure". Returns
    (center [L*Hkv][F][2], mean_norm [L*Hkv][F], mrl [L*Hkv][F]) as float64.
    """
    q = _f64(q)
    L, Hq, n, d = q.shape
    hkv, F = Hq // group, d // 2
    center = np.zeros((L * hkv, F, 2))
    mean_norm = np.zeros((L * hkv, F))
    mrl = np.zeros((L * hkv, F))
    _load().orc_calibrate(_ptr(q), L, Hq, group, n, d, style, _ptr(center), _ptr(mean_norm), _ptr(mrl))
    return center, mean_norm, mrl


def score_series(k, center, mean_norm, mrl, offsets, p_cur: int, theta: float, pos=None,
                 style: int = ROPE_INTERLEAVED, norm_mode: int = NORM_WEIGHTED,
                 return_cos_count: bool = False):
    """Offset-averaged S_trig + S_norm of every row of one slice (TriAttention
    summary page, "The Trigonometric Series Term", "Adaptive Weighting via Q/K
    Concentration", "Handling Multiple Future Positions")."""
    k = _f64(k)
    n, d = k.shape
    pos_a = None if pos is None else _i64(pos)
    offs = _i64(offsets)
    out = np.zeros(n)
    cnt = np.zeros(1, dtype=np.int64)
    _load().orc_score_series(_ptr(k), _ptr(pos_a), n, d, style, float(theta), _ptr(_f64(center)),
                             _ptr(_f64(mean_norm)), _ptr(_f64(mrl)), _ptr(offs), len(offs),
                             int(p_cur), norm_mode, _ptr(out), _ptr(cnt))
    return (out, int(cnt[0])) if return_cos_count else out


def score_bruteforce(k, center, mean_norm, mrl, offsets, p_cur: int, theta: float, pos=None,
                     style: int = ROPE_INTERLEAVED, norm_mode: int = NORM_WEIGHTED):
    """Explicit-rotation form of the same score (TriAttention summary page,
    "The attention dot product in complex form"); tiny inputs only."""
    k = _f64(k)
    n, d = k.shape
    pos_a = None if pos is None else _i64(pos)
    offs = _i64(offsets)
    out = np.zeros(n)
    _load().orc_score_bruteforce(_ptr(k), _ptr(pos_a), n, d, style, float(theta),
                                 _ptr(_f64(center)), _ptr(_f64(mean_norm)), _ptr(_f64(mrl)),
                                 _ptr(offs), len(offs), int(p_cur), norm_mode, _ptr(out))
    return out


def select(score, n_valid: int, n_prompt: int, n_recent: int, budget: int) -> np.ndarray:
    """Protected top-budget keep list, ascending, -1 padded (TriAttention
    summary page, "Retention and eviction"; Random Attention Eq. 2)."""
    s = _f64(score)
    assert s.shape[0] >= n_valid
    keep = np.zeros(budget, dtype=np.int32)
    rc = _load().orc_select(_ptr(s), n_valid, n_prompt, n_recent, budget, _ptr(keep))
    if rc != 0:
        raise ValueError("budget < n_prompt + n_recent")
    return keep


def compact(rows: np.ndarray, keep: np.ndarray) -> int:
    """In-place ascending row gather (Random Attention, Appendix F). rows is
    modified; returns the number of kept rows."""
    assert rows.flags["C_CONTIGUOUS"]
    keep = np.ascontiguousarray(keep, dtype=np.int32)
    row_bytes = rows.nbytes // rows.shape[0]
    return int(_load().orc_compact(_ptr(rows), row_bytes, _ptr(keep), len(keep)))


def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox-4x32-10 of one counter block (Salmon et al., SC'11)."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    kk = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    _load().orc_philox4x32_10(_ptr(c), _ptr(kk), _ptr(out))
    return out


def rand_u32(seed: int, rnd: int, seq: int, layer: int, head: int, slot: int) -> int:
    """The Random Attention draw of one slot, as a 32-bit integer."""
    return int(_load().orc_rand_u32(seed, rnd, seq, layer, head, slot))


def rand_select(seed: int, rnd: int, seq: int, layer: int, head: int, n_valid: int,
                n_prompt: int, n_recent: int, budget: int) -> np.ndarray:
    """Random Attention keep list of one slice (Eq. 3, Algorithm 1)."""
    keep = np.zeros(budget, dtype=np.int32)
    rc = _load().orc_rand_select(seed, rnd, seq, layer, head, n_valid, n_prompt, n_recent,
                                 budget, _ptr(keep))
    if rc != 0:
        raise ValueError("budget < n_prompt + n_recent")
    return keep


def score_bound(k, mean_norm, style: int = ROPE_INTERLEAVED) -> np.ndarray:
    """M(i) = sum_f E|q_f| |k_f|, which bounds |S~(i)| (|E q_f| <= E|q_f|);
    the scale of the score tolerance."""
    k = _f64(k)
    n, d = k.shape
    F = d // 2
    if style == ROPE_INTERLEAVED:
        re, im = k[:, 0::2], k[:, 1::2]
    else:
        re, im = k[:, :F], k[:, F:]
    return np.hypot(re, im) @ _f64(mean_norm)


def score_heads(k, center, mean_norm, mrl, offsets, p_cur: int, theta: float, pos=None,
                style: int = ROPE_INTERLEAVED, norm_mode: int = NORM_WEIGHTED) -> np.ndarray:
    """Scores of one slice under each of the G query heads that share its KV
    head (TriAttention summary page, "Handling Grouped-Query Attention"):
    center [G][F][2], mean_norm and mrl [G][F] are the per-query-head
    statistics. Returns [G][n]."""
    center = _f64(center)
    return np.stack([score_series(k, center[g], mean_norm[g], mrl[g], offsets, p_cur, theta, pos=pos,
                                  style=style, norm_mode=norm_mode) for g in range(center.shape[0])])


def zscore_max(scores_g):
    """Per-head z-score over all cached keys, then the maximum over heads
    (TriAttention summary page, "Handling Grouped-Query Attention").
    scores_g: [G][n]. Returns (mean [G], std [G], final [n])."""
    s = _f64(scores_g)
    G, n = s.shape
    mean, std, final = np.zeros(G), np.zeros(G), np.zeros(n)
    _load().orc_zscore_max(_ptr(s), G, n, _ptr(mean), _ptr(std), _ptr(final))
    return mean, std, final


def rope_rows(x, pos, theta: float, style: int = ROPE_INTERLEAVED, inverse: bool = False) -> np.ndarray:
    """RoPE of every row: row i rotated by omega_f * pos_i, or by -omega_f *
    pos_i when inverse (TriAttention summary page, "RoPE in complex form";
    the blog's invert_rope)."""
    x = _f64(x)
    n, d = x.shape
    p = _i64(pos)
    assert p.shape == (n,)
    out = np.zeros_like(x)
    _load().orc_rope_rows(_ptr(x), _ptr(p), n, d, style, float(theta), -1 if inverse else 1, _ptr(out))
    return out


def score_post_rope(k_post, pos, center, mean_norm, mrl, offsets, p_cur: int, theta: float,
                    style: int = ROPE_INTERLEAVED, norm_mode: int = NORM_WEIGHTED) -> np.ndarray:
    """Score of post-RoPE cached keys (the layout engines keep): undo RoPE with
    each row's position, then the pre-RoPE series (the blog's scoring step)."""
    k = rope_rows(k_post, pos, theta, style=style, inverse=True)
    return score_series(k, center, mean_norm, mrl, offsets, p_cur, theta, pos=pos, style=style,
                        norm_mode=norm_mode)


def rand_select_shared(seed: int, rnd: int, seq: int, layer: int, head: int, scope: int, n_valid: int,
                       n_prompt: int, n_recent: int, budget: int) -> np.ndarray:
    """The shared-draw control of Random Attention (Appendix D): every head
    uses one draw -- head 0's for scope 1 (per layer), layer 0 head 0's for
    scope 2 (per sequence); scope 0 is the per-head draw."""
    if scope >= 1:
        head = 0
    if scope >= 2:
        layer = 0
    return rand_select(seed, rnd, seq, layer, head, n_valid, n_prompt, n_recent, budget)


def union_select(scores_h, n_valid: int, n_prompt: int, n_recent: int, budget: int, k_head: int):
    """One keep list shared by H heads (the blog's union-based selection).
    scores_h: [H][n]. Returns (keep [budget], member [n] bool, combined [n])."""
    s = _f64(scores_h)
    H, n = s.shape
    assert n == n_valid
    member = np.zeros(n, dtype=np.int32)
    combined = np.zeros(n)
    keep = np.zeros(budget, dtype=np.int32)
    rc = _load().orc_union_select(_ptr(s), H, n, n_prompt, n_recent, budget, k_head, _ptr(member),
                                  _ptr(combined), _ptr(keep))
    if rc != 0:
        raise ValueError("budget < n_prompt + n_recent")
    return keep, member.astype(bool), combined


def union_members(scores_h, n_prompt: int, n_recent: int, k_head: int) -> np.ndarray:
    """Step 1 of union_select: the union of every head's top k_head candidates."""
    s = _f64(scores_h)
    H, n = s.shape
    member = np.zeros(n, dtype=np.int32)
    _load().orc_union_members(_ptr(s), H, n, n_prompt, n_recent, k_head, _ptr(member))
    return member.astype(bool)


def union_rank(member, combined, n_prompt: int, n_recent: int, budget: int) -> np.ndarray:
    """Step 2 of union_select: members first by the combined score, then the rest."""
    m = np.ascontiguousarray(np.asarray(member, dtype=np.int32))
    c = _f64(combined)
    keep = np.zeros(budget, dtype=np.int32)
    rc = _load().orc_union_rank(_ptr(m), _ptr(c), len(c), n_prompt, n_recent, budget, _ptr(keep))
    if rc != 0:
        raise ValueError("budget < n_prompt + n_recent")
    return keep
