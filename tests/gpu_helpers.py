"""Shared pieces of the GPU parity tests: run the oracle on chosen slices of
the same inputs the CUDA path consumed, and the comparison rules.

Tolerances (scores to 1e-3 relative, measured against the bound
M(i) = sum_f E|q_f| |k_f| >= |S~(i)|, which keeps the test well posed for
scores near zero):
  scores        |s_gpu - s_ref| <= 1e-3 * M(i)
  selection     the GPU keep set G is valid when |G| = B, protected rows are
                in it, it is ascending, and no kept candidate i and dropped
                candidate j have s_ref(j) - s_ref(i) > 1e-3 * max(M(i), M(j));
                on identical fp32 scores it must equal the oracle bit for bit
  compaction    bytes equal (integer work)
  calibration   |x_gpu - x_ref| <= 1e-5 * E|q_f| per band
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle as orc
import kv_cache_compression_tri_gb300 as tri

SCORE_TOL = 1e-3
CALIB_TOL = 1e-5


def threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def pmap(fn, items):
    with cf.ThreadPoolExecutor(max_workers=threads()) as ex:
        return list(ex.map(fn, items))


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def make_cache(inp, pos: torch.Tensor | None = None, in_place_pos: bool = False) -> tri.KVCache:
    n_seq, L, H, n_cap, d = inp.k.shape
    S = n_seq * L * H
    status = torch.zeros(1, dtype=torch.int32, device=inp.k.device)
    if pos is not None and in_place_pos:
        pos_out = pos
    else:
        pos_out = torch.full((S, n_cap), -7, dtype=torch.int32, device=inp.k.device)
    return tri.KVCache(inp.k, inp.v, inp.n_valid.clone(), pos, pos_out, status)


def slice_rows(t5: torch.Tensor, s: int) -> torch.Tensor:
    n_seq, L, H, n_cap, d = t5.shape
    return t5.view(n_seq * L * H, n_cap, d)[s]


def seq_lh(inp, s: int):
    L, H = inp.k.shape[1], inp.k.shape[2]
    return s // (L * H), s % (L * H)


def oracle_scores(inp, s: int, centers_np, n: int, pos_np=None, style=0, norm_mode=0,
                  offsets=None, p_cur=None):
    """fp64 oracle score and bound M of rows [0, n) of slice s."""
    w = inp.w
    c, m, R = centers_np
    seq, lh = seq_lh(inp, s)
    k = f64(slice_rows(inp.k, s)[:n])
    pc = int(inp.p_cur[seq]) if p_cur is None else int(p_cur)
    offs = w.offsets if offsets is None else offsets
    sref = orc.score_series(k, c[lh], m[lh], R[lh], offs, pc, w.theta, pos=pos_np, style=style,
                            norm_mode=norm_mode)
    M = orc.score_bound(k, m[lh], style=style)
    return sref, M


def near_tie_violations(keep: np.ndarray, s_ref: np.ndarray, M: np.ndarray, n: int, P: int, W: int,
                        B: int, tol: float = SCORE_TOL):
    """Structural checks plus the near-tie rule; returns (problems, swaps)
    where swaps counts kept candidates the oracle would not have kept."""
    problems = []
    keep = np.asarray(keep)
    if n <= B:
        exp = np.concatenate([np.arange(n), -np.ones(B - n, dtype=np.int64)])
        if not np.array_equal(keep, exp):
            problems.append("no-eviction padding differs")
        return problems, 0
    if len(keep) != B or np.any(np.diff(keep) <= 0) or keep.min() < 0 or keep.max() >= n:
        problems.append("keep list not ascending in range")
        return problems, 0
    ks = set(keep.tolist())
    if not set(range(P)) <= ks or not set(range(n - W, n)) <= ks:
        problems.append("protected rows missing")
    cand = np.arange(P, n - W)
    kept_mask = np.zeros(n, dtype=bool)
    kept_mask[keep] = True
    kept = cand[kept_mask[cand]]
    dropped = cand[~kept_mask[cand]]
    if len(kept) != B - P - W:
        problems.append("wrong number of candidates kept")
    if len(dropped) and len(kept):
        order = np.argsort(-s_ref[dropped], kind="stable")
        sd = s_ref[dropped][order]
        ad = (s_ref[dropped] - tol * M[dropped])[order]
        pmax = np.maximum.accumulate(ad)
        thr = s_ref[kept] + tol * M[kept]
        # number of dropped with s_j > thr_i: sd is descending
        cnt = np.searchsorted(-sd, -thr, side="left")
        has = cnt > 0
        viol = has & (pmax[np.maximum(cnt - 1, 0)] > s_ref[kept])
        if np.any(viol):
            problems.append(f"{int(viol.sum())} kept candidates beaten by a dropped one beyond tolerance")
    # swaps relative to the exact oracle ranking
    exact = orc.select(s_ref, n, P, W, B)
    swaps = len(set(exact.tolist()) - ks)
    return problems, swaps
