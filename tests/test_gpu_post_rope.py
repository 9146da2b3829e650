"""GPU parity for caches that hold post-RoPE keys (what engines store; the
TriAttention blog's scoring step inverts RoPE before scoring): the CUDA path
scores the stored keys directly, without positions; the oracle undoes RoPE
with each row's position and runs the pre-RoPE series. Same tolerance as the
pre-RoPE score: |s_gpu - s_ref| <= 1e-3 M(i)."""
import numpy as np
import pytest
import torch

import oracle as orc
import kv_cache_compression_tri_gb300 as tri
from kv_cache_compression_tri_gb300 import synth
from gpu_helpers import SCORE_TOL, f64, make_cache, near_tie_violations, seq_lh, slice_rows

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny"]
LAYER = synth.WORKLOADS["qwen3_8b_layer"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    tri.load_library()


def _post_inputs(w, style, explicit_pos, seed):
    """Pre-RoPE draws of the workload, stored rotated at slot positions or at
    random increasing positions; returns inputs (k post-RoPE) and positions."""
    inp = synth.make_inputs(w, "cuda")
    S, n_cap = w.n_slices, w.n_cap
    rng = np.random.default_rng(seed)
    if explicit_pos:
        pos_np = np.stack([np.sort(rng.choice(4 * n_cap, size=n_cap, replace=False)) for _ in range(S)])
        inp.p_cur = torch.full((w.n_seq,), 4 * n_cap + 5, dtype=torch.int64, device="cuda")
    else:
        pos_np = np.tile(np.arange(n_cap), (S, 1))
    kpre = inp.k.clone()
    for s in range(S):
        rows = slice_rows(inp.k, s)
        rows.copy_(synth.rope_rows(slice_rows(kpre, s).float(), torch.tensor(pos_np[s], device="cuda"),
                                   w.theta, style).to(w.dtype))
    return inp, kpre, pos_np


def _post_case(w, style=0, norm_mode=0, explicit_pos=False, ragged=False, seed=0):
    inp, kpre, pos_np = _post_inputs(w, style, explicit_pos, seed)
    S, n_cap = w.n_slices, w.n_cap
    c = tri.calibrate_centers(inp.q, w.group, style=style)
    if ragged:
        rng = np.random.default_rng(seed + 100)
        nv = rng.integers(0, n_cap + 1, size=S)
        nv[0], nv[-1] = n_cap, 1
        inp.n_valid = torch.tensor(nv, dtype=torch.int32, device="cuda")
    # positions are handed over (compaction would move them) but the score must not need them
    pos = torch.tensor(pos_np, dtype=torch.int32, device="cuda") if explicit_pos else None
    kv = make_cache(inp, pos=pos)
    kv.post_rope = True
    scores = torch.full((S, n_cap), 12345.0, device="cuda")
    tri.score(kv, c, w.theta, w.offsets, inp.p_cur, scores, style=style, norm_mode=norm_mode)
    # the same keys before RoPE, scored as pre-RoPE keys with their positions
    kv_pre = make_cache(inp, pos=torch.tensor(pos_np, dtype=torch.int32, device="cuda"))
    kv_pre.k = kpre
    scores_pre = torch.full((S, n_cap), 12345.0, device="cuda")
    tri.score(kv_pre, c, w.theta, w.offsets, inp.p_cur, scores_pre, style=style, norm_mode=norm_mode)
    torch.cuda.synchronize()
    assert int(kv.dev_status.item()) == 0
    cc, cm, cR = f64(c.center), f64(c.mean_norm), f64(c.mrl)
    g, gp = scores.cpu().numpy(), scores_pre.cpu().numpy()
    nvh = kv.n_valid.cpu().numpy()
    worst = 0.0
    for s in range(S):
        n = int(nvh[s])
        seq, lh = seq_lh(inp, s)
        kpost = f64(slice_rows(inp.k, s)[:n])
        ref = orc.score_post_rope(kpost, pos_np[s, :n], cc[lh], cm[lh], cR[lh], w.offsets, int(inp.p_cur[seq]),
                                  w.theta, style=style, norm_mode=norm_mode)
        M = orc.score_bound(kpost, cm[lh], style=style)
        if n:
            err = np.abs(g[s, :n] - ref) / M
            worst = max(worst, float(err.max()))
            assert np.all(err <= SCORE_TOL), (s, float(err.max()))
            # the pre-RoPE draws give the same scores up to the bf16 rounding of
            # the rotated copy: both within the tolerance of their own oracle
            kp = f64(slice_rows(kpre, s)[:n])
            ref_pre = orc.score_series(kp, cc[lh], cm[lh], cR[lh], w.offsets, int(inp.p_cur[seq]), w.theta,
                                       pos=pos_np[s, :n], style=style, norm_mode=norm_mode)
            assert np.all(np.abs(gp[s, :n] - ref_pre) <= SCORE_TOL * M)
        assert np.all(g[s, n:] == 12345.0)
    return worst


@pytest.mark.parametrize("style", [0, 1])
def test_post_rope_score_layer(style):
    assert _post_case(LAYER, style=style) < 1e-4


def test_post_rope_score_explicit_positions_and_ragged():
    _post_case(LAYER, explicit_pos=True, ragged=True, seed=3)
    w1 = synth.scaled(TINY, dtype=torch.bfloat16, n_seq=2, n_layers=2, n_kv_heads=2, group=2, n_cap=1000,
                      n_valid=1000, n_cal=512)
    _post_case(w1, style=1, explicit_pos=True, seed=4)
    _post_case(w1, norm_mode=1, ragged=True, seed=5)
    w2 = synth.scaled(LAYER, dtype=torch.float32, n_kv_heads=2, n_cap=700, n_valid=700, n_cal=256)
    _post_case(w2, style=0, explicit_pos=True, seed=6)
    _post_case(w2, style=1, seed=7)


def test_post_rope_gqa_heads_and_selection():
    w = synth.scaled(LAYER, n_kv_heads=4, n_cap=1500, n_valid=1500, n_cal=512, n_prompt=64, n_recent=32,
                     budget=500)
    G = w.group
    inp, kpre, pos_np = _post_inputs(w, 0, True, 11)
    S, n_cap = w.n_slices, w.n_cap
    cq = tri.calibrate_centers(inp.q, 1)
    kv = make_cache(inp, pos=torch.tensor(pos_np, dtype=torch.int32, device="cuda"))
    kv.post_rope = True
    scores_g = torch.full((S, G, n_cap), 12345.0, device="cuda")
    stats = torch.empty(S, G, 2, device="cuda")
    tri.score_heads(kv, cq, G, w.theta, w.offsets, inp.p_cur, scores_g, stats)
    keep = torch.empty(S, w.budget, dtype=torch.int32, device="cuda")
    final = torch.empty(S, n_cap, device="cuda")
    tri.select_topk_zmax(scores_g, stats, G, kv, w.n_prompt, w.n_recent, w.budget, keep, final_scores=final)
    torch.cuda.synchronize()
    assert int(kv.dev_status.item()) == 0
    c, m, R = f64(cq.center), f64(cq.mean_norm), f64(cq.mrl)
    g_sc, g_fin, g_keep = scores_g.cpu().numpy(), final.cpu().numpy(), keep.cpu().numpy()
    for s in range(S):
        seq, lh = seq_lh(inp, s)
        kpost = f64(slice_rows(inp.k, s))
        kpre_rows = orc.rope_rows(kpost, pos_np[s], w.theta, inverse=True)
        rows = slice(lh * G, (lh + 1) * G)
        ref = orc.score_heads(kpre_rows, c[rows], m[rows], R[rows], w.offsets, int(inp.p_cur[seq]), w.theta,
                              pos=pos_np[s])
        Mg = np.stack([orc.score_bound(kpost, m[lh * G + g]) for g in range(G)])
        assert np.all(np.abs(g_sc[s] - ref) <= SCORE_TOL * Mg), s
        assert np.array_equal(g_keep[s], orc.select(g_fin[s].astype(np.float64), n_cap, w.n_prompt, w.n_recent,
                                                    w.budget)), s
