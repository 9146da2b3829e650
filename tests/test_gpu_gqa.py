"""GPU parity of the GQA path -- one score per query head, the per-head
statistics over all cached keys, and the selection by the maximum z-score
(TriAttention summary page, "Handling Grouped-Query Attention") -- through
the C ABI, against the fp64 oracle on the same seeded inputs.

Tolerances follow from the score tolerance |s_gpu - s_ref| <= 1e-3 M_g(i)
(M_g(i) = sum_f E|q(g)_f| |k_f|, the bound on head g's score):
  mean, std of head g   <= 1e-3 max_i M_g(i)   (a mean moves by at most the
                           largest score error, a standard deviation by at
                           most their root mean square)
  final score           <= 1e-3 max_g (M_g(i) + 2 max M_g (1 + |z_g(i)|)) / std_g
The selection must equal the oracle's selection run on the GPU's own fp32
final scores bit for bit, and obey the near-tie rule against the oracle's
fp64 final scores.
"""
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


def _heads_case(w, style=0, norm_mode=0, explicit_pos=False, ragged=False, P=None, W=None, B=None,
                zero_slice=None, seed=0):
    G = w.group
    inp = synth.make_inputs(w, "cuda")
    S, n_cap = w.n_slices, w.n_cap
    P = w.n_prompt if P is None else P
    W = w.n_recent if W is None else W
    B = w.budget if B is None else B
    cq = tri.calibrate_centers(inp.q, 1, style=style)  # one row per query head
    rng = np.random.default_rng(seed)
    if ragged:
        nv = rng.integers(0, n_cap + 1, size=S)
        nv[0], nv[-1] = n_cap, 1
        if S > 2:
            nv[1] = 0
        inp.n_valid = torch.tensor(nv, dtype=torch.int32, device="cuda")
    if zero_slice is not None:
        slice_rows(inp.k, zero_slice).zero_()  # every head scores every key alike
    pos = None
    if explicit_pos:
        pos_np = np.stack([np.sort(rng.choice(4 * n_cap, size=n_cap, replace=False)) for _ in range(S)])
        pos = torch.tensor(pos_np, dtype=torch.int32, device="cuda")
        inp.p_cur = torch.full((w.n_seq,), 4 * n_cap + 5, dtype=torch.int64, device="cuda")
    kv = make_cache(inp, pos=pos)
    scores_g = torch.full((S, G, n_cap), 12345.0, device="cuda")
    stats = torch.full((S, G, 2), -1.0, device="cuda")
    n0 = tri.launch_count()
    tri.score_heads(kv, cq, G, w.theta, w.offsets, inp.p_cur, scores_g, stats, style=style,
                    norm_mode=norm_mode)
    per_pass = 8 if w.dtype == torch.bfloat16 else 4  # tensor-core kernel for bf16 keys
    assert tri.launch_count() - n0 == (G + per_pass - 1) // per_pass + 1  # score passes + statistics
    keep = torch.full((S, B), -9, dtype=torch.int32, device="cuda")
    final = torch.full((S, n_cap), 777.0, device="cuda")
    tri.select_topk_zmax(scores_g, stats, G, kv, P, W, B, keep, final_scores=final)
    torch.cuda.synchronize()
    assert int(kv.dev_status.item()) == 0

    c, m, R = f64(cq.center), f64(cq.mean_norm), f64(cq.mrl)
    g_sc, g_st, g_keep, g_fin = scores_g.cpu().numpy(), stats.cpu().numpy(), keep.cpu().numpy(), \
        final.cpu().numpy()
    nvh = kv.n_valid.cpu().numpy()
    worst = 0.0
    for s in range(S):
        n = int(nvh[s])
        seq, lh = seq_lh(inp, s)
        rows = slice(lh * G, (lh + 1) * G)
        k = f64(slice_rows(inp.k, s)[:n])
        pos_s = None if pos is None else pos[s, :n].cpu().numpy().astype(np.int64)
        ref = orc.score_heads(k, c[rows], m[rows], R[rows], w.offsets, int(inp.p_cur[seq]), w.theta,
                              pos=pos_s, style=style, norm_mode=norm_mode)
        Mg = np.stack([orc.score_bound(k, m[lh * G + g], style=style) for g in range(G)]) if n else \
            np.zeros((G, 0))
        # per-head scores, and rows >= n untouched
        if n:
            err = np.abs(g_sc[s, :, :n] - ref) / np.maximum(Mg, 1e-30)
            worst = max(worst, float(err.max()))
            assert np.all(err <= SCORE_TOL), (s, float(err.max()))
        assert np.all(g_sc[s, :, n:] == 12345.0)
        # statistics
        mu, sd, fin = orc.zscore_max(ref) if n else (np.zeros(G), np.zeros(G), np.zeros(0))
        mmax = Mg.max(axis=1) if n else np.zeros(G)
        tol_st = SCORE_TOL * mmax + 1e-6 * (np.abs(mu) + sd)
        assert np.all(np.abs(g_st[s, :, 0] - mu) <= tol_st), (s, g_st[s, :, 0], mu)
        assert np.all(np.abs(g_st[s, :, 1] - sd) <= tol_st), (s, g_st[s, :, 1], sd)
        if n == 0:
            assert np.all(g_st[s] == 0.0)
            continue
        # final scores: the GPU's own arithmetic on its own scores and statistics ...
        gm, gs = g_st[s, :, 0].astype(np.float64), g_st[s, :, 1].astype(np.float64)
        inv = np.where(gs > 0, 1.0 / np.where(gs > 0, gs, 1.0), 0.0)
        own = ((g_sc[s, :, :n].astype(np.float64) - gm[:, None]) * inv[:, None]).max(axis=0)
        assert np.all(np.abs(g_fin[s, :n] - own) <= 1e-5 * (1.0 + np.abs(own))), s
        assert np.all(g_fin[s, n:] == 777.0)
        # ... and against the oracle within the propagated tolerance
        z = np.where(sd[:, None] > 0, (ref - mu[:, None]) / np.where(sd > 0, sd, 1.0)[:, None], 0.0)
        tol_z = np.where(sd[:, None] > 0,
                         SCORE_TOL * (Mg + 2 * mmax[:, None] * (1 + np.abs(z))) / np.where(sd > 0, sd, 1.0)[:, None],
                         0.0).max(axis=0) + 1e-6
        assert np.all(np.abs(g_fin[s, :n] - fin) <= tol_z), s
        # selection: bit-exact on the GPU's fp32 final scores, near ties vs fp64
        assert np.array_equal(g_keep[s], orc.select(g_fin[s, :n].astype(np.float64), n, P, W, B)), s
        problems, _ = near_tie_violations(g_keep[s], fin, tol_z, n, P, W, B, tol=1.0)
        assert not problems, (s, problems)
    return worst


def test_gqa_layer_workload():
    worst = _heads_case(LAYER)
    assert worst < 1e-4


@pytest.mark.parametrize("group", [1, 2, 3, 7, 8])
def test_gqa_group_sizes(group):
    # bf16 keys: one pass over K for up to eight heads (tensor cores)
    w = synth.scaled(LAYER, group=group, n_kv_heads=2, n_layers=2, n_cap=1000, n_valid=1000, n_cal=512,
                     n_prompt=40, n_recent=24, budget=300)
    _heads_case(w, seed=group)


@pytest.mark.parametrize("group", [4, 8])
def test_gqa_bf16_d128_runs_of_one_to_three_blocks(group):
    # 300-row caches: a CTA's run is one to three 128-row blocks (the second
    # group of feature warps idle, or the third operand buffer unused), with
    # ragged row counts 0, 1 and in between
    w = synth.scaled(LAYER, group=group, n_kv_heads=2, n_layers=3, n_cap=300, n_valid=300, n_cal=256,
                     n_prompt=8, n_recent=8, budget=64)
    _heads_case(w, ragged=True, seed=10 + group)


def test_gqa_bf16_d64_and_fp32_d128():
    w1 = synth.scaled(TINY, dtype=torch.bfloat16, n_seq=2, n_layers=2, n_kv_heads=2, group=4, n_cap=1000,
                      n_valid=1000, n_cal=512, n_prompt=16, n_recent=16, budget=250)
    _heads_case(w1, ragged=True, seed=1)
    _heads_case(w1, style=1, explicit_pos=True, seed=2)
    w2 = synth.scaled(LAYER, dtype=torch.float32, n_kv_heads=2, n_cap=700, n_valid=700, n_cal=256,
                      n_prompt=30, n_recent=10, budget=200)
    _heads_case(w2, norm_mode=1, ragged=True, seed=3)
    _heads_case(w2, style=1, explicit_pos=True, seed=4)


def test_gqa_constant_scores_and_no_eviction():
    # all-zero keys: every head scores 0 everywhere, std 0, final 0, lowest slots win
    w = synth.scaled(LAYER, n_kv_heads=2, n_cap=600, n_valid=600, n_cal=256, n_prompt=8, n_recent=8, budget=100)
    _heads_case(w, zero_slice=1)
    _heads_case(w, B=600)  # n_valid == budget: nothing evicted


def test_gqa_bf16_band_beyond_fp16_range_is_reported():
    # bf16 keys go through fp16 features: a band of magnitude >= 65520 has no
    # fp16 value, its scores come out non-finite and the selection says so
    w = synth.scaled(LAYER, n_kv_heads=2, n_cap=600, n_valid=600, n_cal=256, n_prompt=8, n_recent=8, budget=100)
    inp = synth.make_inputs(w, "cuda")
    cq = tri.calibrate_centers(inp.q, 1)
    slice_rows(inp.k, 1)[300, 0:2] = 2.0e5
    kv = make_cache(inp)
    S, G = w.n_slices, w.group
    scores_g = torch.zeros(S, G, w.n_cap, device="cuda")
    stats = torch.zeros(S, G, 2, device="cuda")
    tri.score_heads(kv, cq, G, w.theta, w.offsets, inp.p_cur, scores_g, stats)
    keep = torch.empty(S, w.budget, dtype=torch.int32, device="cuda")
    tri.select_topk_zmax(scores_g, stats, G, kv, w.n_prompt, w.n_recent, w.budget, keep)
    torch.cuda.synchronize()
    assert int(kv.dev_status.item()) == tri.DEV_NAN_SCORE
    assert torch.isfinite(scores_g[0]).all()  # the other slice is untouched by it


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_gqa_repeated_launches_are_bit_identical(dtype):
    # A whole 36-layer sequence (576 CTAs of the tensor-core kernel, every SM
    # busy and HBM loaded): ten launches give the same bits and no device
    # error. A pipeline whose stages were handed over out of order would read
    # tiles or accumulators mid-flight and differ from run to run.
    w = synth.scaled(synth.WORKLOADS["qwen3_8b_stack"], n_seq=1, dtype=dtype, n_cal=256)
    inp = synth.make_inputs(w, "cuda")
    cq = tri.calibrate_centers(inp.q, 1)
    inp.q = None
    kv = make_cache(inp)
    S, G = w.n_slices, w.group
    runs = []
    for _ in range(10):
        scores_g = torch.full((S, G, w.n_cap), 12345.0, device="cuda")
        stats = torch.full((S, G, 2), -1.0, device="cuda")
        tri.score_heads(kv, cq, G, w.theta, w.offsets, inp.p_cur, scores_g, stats)
        torch.cuda.synchronize()
        assert int(kv.dev_status.item()) == 0
        runs.append((scores_g, stats))
    s0, t0 = runs[0]
    assert torch.isfinite(s0).all() and torch.isfinite(t0).all()
    for s1, t1 in runs[1:]:
        assert torch.equal(s1, s0) and torch.equal(t1, t0)
