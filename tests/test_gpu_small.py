"""GPU parity on the small workloads (every slice) and on edge cases, through
the C ABI, against the fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle as orc
import kv_cache_compression_tri_gb300 as tri
from kv_cache_compression_tri_gb300 import synth
from gpu_helpers import (CALIB_TOL, SCORE_TOL, f64, make_cache, near_tie_violations, oracle_scores,
                         pmap, seq_lh, slice_rows)

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny"]
LAYER = synth.WORKLOADS["qwen3_8b_layer"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    tri.load_library()


def _centers_np(c: tri.Centers):
    return (f64(c.center), f64(c.mean_norm), f64(c.mrl))


@pytest.mark.parametrize("wname", ["tiny", "qwen3_8b_layer"])
@pytest.mark.parametrize("style", [0, 1])
def test_calibrate_parity(wname, style):
    w = synth.WORKLOADS[wname]
    inp = synth.make_inputs(w, "cuda")
    c = tri.calibrate_centers(inp.q, w.group, style=style)
    torch.cuda.synchronize()
    rc, rm, rR = orc.calibrate(f64(inp.q), w.group, style=style)
    gc, gm, gR = _centers_np(c)
    scale = rm[..., None]
    assert np.all(np.abs(gc - rc) <= CALIB_TOL * scale)
    assert np.all(np.abs(gm - rm) <= CALIB_TOL * rm)
    assert np.all(np.abs(gR - rR) <= CALIB_TOL)


def _score_case(w, style=0, norm_mode=0, explicit_pos=False, ragged=False, P=0, W=0, seed=0):
    inp = synth.make_inputs(w, "cuda")
    S, n_cap = w.n_slices, w.n_cap
    c = tri.calibrate_centers(inp.q, w.group, style=style)
    rng = np.random.default_rng(seed)
    if ragged:
        nv = rng.integers(0, n_cap + 1, size=S)
        nv[0], nv[-1] = n_cap, 1
        inp.n_valid = torch.tensor(nv, dtype=torch.int32, device="cuda")
    pos = None
    if explicit_pos:
        pos_np = np.stack([np.sort(rng.choice(4 * n_cap, size=n_cap, replace=False)) for _ in range(S)])
        pos = torch.tensor(pos_np, dtype=torch.int32, device="cuda")
        inp.p_cur = torch.full((w.n_seq,), 4 * n_cap + 5, dtype=torch.int64, device="cuda")
    kv = make_cache(inp, pos=pos)
    scores = torch.full((S, n_cap), 12345.0, device="cuda")
    tri.score(kv, c, w.theta, w.offsets, inp.p_cur, scores, n_prompt=P, n_recent=W, style=style,
              norm_mode=norm_mode)
    torch.cuda.synchronize()
    cn = _centers_np(c)
    g = scores.cpu().numpy()
    nvh = kv.n_valid.cpu().numpy()
    worst = 0.0
    for s in range(S):
        n = int(nvh[s])
        pos_np_s = None if pos is None else pos[s, :n].cpu().numpy().astype(np.int64)
        sref, M = oracle_scores(inp, s, cn, n, pos_np=pos_np_s, style=style, norm_mode=norm_mode)
        lo, hi = P, max(n - W, P)
        err = np.abs(g[s, lo:hi] - sref[lo:hi]) / M[lo:hi]
        if len(err):
            worst = max(worst, float(err.max()))
        assert np.all(err <= SCORE_TOL), (s, float(err.max()))
        # rows outside [P, n - W) are not written
        untouched = np.concatenate([g[s, :lo], g[s, max(hi, lo):]])
        assert np.all(untouched == 12345.0)
    assert int(kv.dev_status.item()) == 0
    return worst


@pytest.mark.parametrize("wname", ["tiny", "qwen3_8b_layer"])
@pytest.mark.parametrize("style", [0, 1])
def test_score_parity_all_rows(wname, style):
    worst = _score_case(synth.WORKLOADS[wname], style=style)
    assert worst < 1e-4  # far inside the tolerance: fp32 rounding only


def test_score_parity_protected_rows_skipped():
    _score_case(TINY, P=32, W=64)
    _score_case(LAYER, P=256, W=128)


@pytest.mark.parametrize("wname", ["tiny", "qwen3_8b_layer"])
def test_score_parity_explicit_positions(wname):
    _score_case(synth.WORKLOADS[wname], explicit_pos=True, seed=3)


def test_score_parity_unweighted_norm_and_ragged():
    _score_case(LAYER, norm_mode=1, ragged=True, seed=5)
    _score_case(synth.scaled(LAYER, n_seq=3, n_layers=2), ragged=True, seed=6, P=7, W=9)


def test_score_parity_bf16_d64_and_fp32_d128():
    w1 = synth.scaled(TINY, dtype=torch.bfloat16, n_seq=2, n_layers=3, n_kv_heads=4, group=2,
                      n_cap=1000, n_valid=1000, n_cal=512)
    _score_case(w1, ragged=True, seed=8)
    _score_case(w1, style=1, explicit_pos=True, seed=9)
    w2 = synth.scaled(LAYER, dtype=torch.float32, n_kv_heads=2, n_cap=700, n_valid=700, n_cal=256)
    _score_case(w2, style=1, seed=10)
    _score_case(w2, style=0, explicit_pos=True, seed=11)


def _select_case(S, n_cap, P, W, B, n_valid, scores_np, nan_expected=False):
    dev = "cuda"
    k = torch.zeros(1, 1, S, n_cap, 64, dtype=torch.bfloat16, device=dev)
    kv = tri.KVCache(k, k, torch.tensor(n_valid, dtype=torch.int32, device=dev), None, None,
                     torch.zeros(1, dtype=torch.int32, device=dev))
    sc = torch.tensor(scores_np, dtype=torch.float32, device=dev)
    keep = torch.full((S, B), -9, dtype=torch.int32, device=dev)
    tri.select_topk(sc, kv, P, W, B, keep)
    torch.cuda.synchronize()
    g = keep.cpu().numpy()
    for s in range(S):
        exp = orc.select(scores_np[s].astype(np.float32).astype(np.float64), int(n_valid[s]), P, W, B)
        assert np.array_equal(g[s], exp), s
    assert int(kv.dev_status.item()) == (tri.DEV_NAN_SCORE if nan_expected else 0)


@pytest.mark.parametrize("seed", range(3))
def test_select_bit_exact_with_ties(seed):
    rng = np.random.default_rng(seed)
    S, n_cap = 6, 5000
    sc = np.round(rng.normal(size=(S, n_cap)) * 4) / 4  # heavy exact ties
    sc[0] = 1.0  # all equal
    sc[1, ::7] = -0.0
    sc[1, 1::7] = 0.0
    sc[2, :100] = np.inf
    sc[3, 50:60] = -np.inf
    nv = [5000, 4999, 4000, 300, 100, 5000]
    _select_case(S, n_cap, 17, 33, 300, nv, sc.astype(np.float32))


def test_select_nan_ranks_lowest():
    rng = np.random.default_rng(9)
    sc = rng.normal(size=(2, 3000)).astype(np.float32)
    sc[0, 100:2000] = np.nan
    _select_case(2, 3000, 10, 10, 1500, [3000, 3000], sc, nan_expected=True)


def test_select_degenerate_budgets():
    rng = np.random.default_rng(2)
    sc = rng.normal(size=(3, 1000)).astype(np.float32)
    _select_case(3, 1000, 100, 100, 200, [1000, 201, 200], sc)  # nothing to select / n == B
    _select_case(3, 1000, 0, 0, 1, [1000, 1000, 0], sc)  # B = 1, empty slice
    _select_case(3, 1000, 0, 0, 999, [1000, 1000, 1000], sc)  # drop one


def test_select_streaming_super_chunks():
    # more candidates than the bitmaps cover: they are rebuilt piece by piece
    rng = np.random.default_rng(4)
    n_cap = 70001
    sc = (np.round(rng.normal(size=(2, n_cap)) * 64) / 64).astype(np.float32)
    _select_case(2, n_cap, 3, 5, 20000, [n_cap, 65536 + 77], sc)


def test_select_sampled_window_full_length():
    # 32K candidates of continuous scores: the window comes from a sample
    rng = np.random.default_rng(11)
    n_cap = 32768
    sc = rng.normal(size=(4, n_cap)).astype(np.float32)
    sc[1] += np.linspace(0, 3, n_cap, dtype=np.float32)  # a trend along the slots
    sc[2] = np.abs(sc[2]) ** 3  # heavy tail
    _select_case(4, n_cap, 512, 128, 4096, [n_cap, n_cap, n_cap - 5, 20000], sc)
    _select_case(4, n_cap, 0, 0, 7, [n_cap] * 4, sc)  # tiny need
    _select_case(4, n_cap, 8, 8, n_cap - 40, [n_cap] * 4, sc)  # keep almost all


def test_select_threshold_ties_overflow_the_list():
    # 6000 candidates tie at the threshold: more than the short list holds,
    # so the exact selection over all candidates decides; lower slots win
    rng = np.random.default_rng(12)
    n_cap = 10000
    sc = np.full((2, n_cap), 0.5, dtype=np.float32)
    perm = rng.permutation(n_cap)
    sc[0, perm[:2000]] = 2.0 + rng.random(2000)
    sc[0, perm[2000:4000]] = -rng.random(2000)
    sc[1] = sc[0][::-1]
    _select_case(2, n_cap, 0, 0, 3000, [n_cap, n_cap], sc)


def test_select_sample_misled_by_layout():
    # every 20th slot (where a systematic sample of 2048 of 40960 candidates
    # lands) is far below the rest, so any window drawn from those slots is
    # wrong; the result must still be exact
    rng = np.random.default_rng(13)
    n_cap, P = 40960 + 64, 64
    sc = rng.normal(size=(2, n_cap)).astype(np.float32)
    sc[:, P + 10::20] -= 10.0
    sc[1, P + 10::20] += 20.0  # or far above it
    _select_case(2, n_cap, P, 0, 4000, [n_cap, n_cap], sc)


def _compact_case(w, keep_np, pos_mode="none", seed=0):
    inp = synth.make_inputs(w, "cuda", with_queries=False)
    S, n_cap = w.n_slices, w.n_cap
    B = keep_np.shape[1]
    pos = None
    if pos_mode != "none":
        rng = np.random.default_rng(seed)
        pos = torch.tensor(np.sort(rng.integers(0, 1 << 30, size=(S, n_cap)), axis=1), dtype=torch.int32,
                           device="cuda")
    pristine_k = inp.k.clone()
    pristine_v = inp.v.clone()
    pristine_pos = None if pos is None else pos.clone()
    kv = make_cache(inp, pos=pos, in_place_pos=(pos_mode == "inplace"))
    keep = torch.tensor(keep_np, dtype=torch.int32, device="cuda")
    tri.compact_kv(kv, keep, B)
    torch.cuda.synchronize()
    assert int(kv.dev_status.item()) == 0
    d = w.head_dim
    for s in range(S):
        for cur, pr in ((kv.k, pristine_k), (kv.v, pristine_v)):
            rows = slice_rows(pr, s).cpu().contiguous().view(torch.uint8).numpy().reshape(n_cap, -1).copy()
            n_keep = orc.compact(rows, keep_np[s])
            got = slice_rows(cur, s).cpu().contiguous().view(torch.uint8).numpy().reshape(n_cap, -1)
            assert np.array_equal(got, rows), s
        n_keep = int(np.argmax(keep_np[s] < 0)) if (keep_np[s] < 0).any() else B
        assert int(kv.n_valid[s]) == n_keep
        po = kv.pos_out[s].cpu().numpy()
        src = keep_np[s][:n_keep]
        if pristine_pos is None:
            assert np.array_equal(po[:n_keep], src)
        else:
            assert np.array_equal(po[:n_keep], pristine_pos[s].cpu().numpy()[src])
            if pos_mode == "inplace":
                assert np.array_equal(po[n_keep:], pristine_pos[s].cpu().numpy()[n_keep:])


def _keeps(S, n_cap, B, rng):
    ks = []
    for s in range(S):
        kind = s % 5
        if kind == 0:
            k = np.sort(rng.choice(n_cap, size=B, replace=False))
        elif kind == 1:
            k = np.arange(1, B + 1)  # every source is overwritten later: in-place hazard
        elif kind == 2:
            k = np.arange(n_cap - B, n_cap)
        elif kind == 3:
            k = np.concatenate([np.arange(B // 2), np.sort(rng.choice(np.arange(B // 2, n_cap), B - B // 2, replace=False))])
        else:
            n = int(rng.integers(0, B))
            k = np.concatenate([np.arange(n), -np.ones(B - n, dtype=np.int64)])
        ks.append(k)
    return np.stack(ks).astype(np.int32)


@pytest.mark.parametrize("pos_mode", ["none", "gather", "inplace"])
def test_compact_bit_exact(pos_mode):
    w = synth.scaled(LAYER, n_kv_heads=10, n_cap=3000, n_valid=3000)
    rng = np.random.default_rng(1)
    _compact_case(w, _keeps(10, 3000, 1000, rng), pos_mode=pos_mode)
    w2 = synth.scaled(TINY, n_kv_heads=5, n_cap=700, n_valid=700, dtype=torch.bfloat16)
    _compact_case(w2, _keeps(5, 700, 300, rng), pos_mode=pos_mode)
    w3 = synth.scaled(TINY, n_kv_heads=5, n_cap=700, n_valid=700)  # fp32, d 64
    _compact_case(w3, _keeps(5, 700, 257, rng), pos_mode=pos_mode)


def test_compact_rejects_malformed_keep_without_touching_cache():
    w = synth.scaled(TINY, n_kv_heads=3, n_cap=300, n_valid=300, dtype=torch.bfloat16)
    inp = synth.make_inputs(w, "cuda", with_queries=False)
    before = inp.k.clone()
    kv = make_cache(inp)
    keep = torch.tensor(np.stack([np.arange(1, 101), np.r_[np.arange(50), np.arange(40, 90)],
                                  np.r_[np.arange(99), [300]]]), dtype=torch.int32, device="cuda")
    tri.compact_kv(kv, keep, 100)
    torch.cuda.synchronize()
    assert int(kv.dev_status.item()) == tri.DEV_BAD_KEEP
    # slice 0 is valid and compacted; slices 1 (descending) and 2 (out of range) untouched
    assert torch.equal(slice_rows(inp.k, 1), slice_rows(before, 1))
    assert torch.equal(slice_rows(inp.k, 2), slice_rows(before, 2))
    assert torch.equal(slice_rows(inp.k, 0)[:100], slice_rows(before, 0)[1:101])


@pytest.mark.parametrize("P,W", [(0, 0), (13, 0), (512, 64), (3, 7)])
def test_random_bit_exact(P, W):
    w = synth.scaled(LAYER, n_seq=2, n_layers=3, n_kv_heads=4, n_cap=6000, n_valid=6000)
    S = w.n_slices
    nv = np.full(S, 6000)
    nv[1], nv[2], nv[3] = 1500, 1499, 5999
    # the random path never reads K/V; the cache only fixes shapes
    k = torch.zeros(w.n_seq, w.n_layers, w.n_kv_heads, 6000, 64, dtype=torch.bfloat16, device="cuda")
    kv = tri.KVCache(k, k, torch.tensor(nv, dtype=torch.int32, device="cuda"), None, None,
                     torch.zeros(1, dtype=torch.int32, device="cuda"))
    B = 1500
    for rnd in (0, 7):
        keep = torch.full((S, B), -9, dtype=torch.int32, device="cuda")
        tri.rand_evict(kv, 0xC0FFEE1234, rnd, P, W, B, keep)
        torch.cuda.synchronize()
        g = keep.cpu().numpy()
        for s in range(S):
            seq, rem = divmod(s, w.n_layers * w.n_kv_heads)
            layer, head = divmod(rem, w.n_kv_heads)
            exp = orc.rand_select(0xC0FFEE1234, rnd, seq, layer, head, int(nv[s]), P, W, B)
            assert np.array_equal(g[s], exp), (rnd, s)


@pytest.mark.parametrize("scope", [1, 2])
def test_random_shared_draw(scope):
    # Random Attention's shared-draw control: one keep-set for every head of a
    # layer (scope 1) or of a sequence (scope 2)
    w = synth.scaled(LAYER, n_seq=2, n_layers=3, n_kv_heads=4, n_cap=6000, n_valid=6000)
    S = w.n_slices
    k = torch.zeros(w.n_seq, w.n_layers, w.n_kv_heads, 6000, 64, dtype=torch.bfloat16, device="cuda")
    kv = tri.KVCache(k, k, torch.full((S,), 6000, dtype=torch.int32, device="cuda"), None, None,
                     torch.zeros(1, dtype=torch.int32, device="cuda"))
    B, P = 1500, 100
    keep = torch.full((S, B), -9, dtype=torch.int32, device="cuda")
    tri.rand_evict_scoped(kv, 0xABCDEF, 5, scope, P, 0, B, keep)
    torch.cuda.synchronize()
    g = keep.cpu().numpy()
    for s in range(S):
        seq, rem = divmod(s, w.n_layers * w.n_kv_heads)
        layer, head = divmod(rem, w.n_kv_heads)
        exp = orc.rand_select_shared(0xABCDEF, 5, seq, layer, head, scope, 6000, P, 0, B)
        assert np.array_equal(g[s], exp), s
        first = seq * w.n_layers * w.n_kv_heads + (0 if scope == 2 else layer * w.n_kv_heads)
        assert np.array_equal(g[s], g[first])
    # per-head draws differ from head to head
    tri.rand_evict_scoped(kv, 0xABCDEF, 5, 0, P, 0, B, keep)
    torch.cuda.synchronize()
    g0 = keep.cpu().numpy()
    assert not np.array_equal(g0[0], g0[1])


@pytest.mark.parametrize("scope", [0, 1])
def test_rand_evict_compact_equals_two_calls(scope):
    w = synth.scaled(LAYER, n_seq=2, n_layers=2, n_kv_heads=4, n_cap=3000, n_valid=3000)
    inp = synth.make_inputs(w, "cuda", with_queries=False)
    S = w.n_slices
    nv = np.random.default_rng(8).integers(0, 3001, size=S)
    nv[0] = 3000
    k0, v0 = inp.k.clone(), inp.v.clone()
    out = []
    for fused in (False, True):
        kv = tri.KVCache(k0.clone(), v0.clone(), torch.tensor(nv, dtype=torch.int32, device="cuda"), None,
                         torch.zeros(S, 3000, dtype=torch.int32, device="cuda"),
                         torch.zeros(1, dtype=torch.int32, device="cuda"))
        keep = torch.full((S, 900), -5, dtype=torch.int32, device="cuda")
        if fused:
            tri.rand_evict_compact(kv, 1234, 2, 100, 0, 900, keep, scope=scope)
        else:
            tri.rand_evict_scoped(kv, 1234, 2, scope, 100, 0, 900, keep)
            tri.compact_kv(kv, keep, 900)
        torch.cuda.synchronize()
        assert int(kv.dev_status.item()) == 0
        out.append((keep, kv))
    (ka, a), (kb, b) = out
    assert torch.equal(ka, kb) and torch.equal(a.k, b.k) and torch.equal(a.v, b.v)
    assert torch.equal(a.n_valid, b.n_valid) and torch.equal(a.pos_out, b.pos_out)


def test_nvalid_over_capacity_sets_status():
    w = synth.scaled(TINY, n_kv_heads=2, n_cap=256, n_valid=256, dtype=torch.bfloat16)
    inp = synth.make_inputs(w, "cuda")
    c = tri.calibrate_centers(inp.q, w.group)
    kv = make_cache(inp)
    kv.n_valid[1] = 300
    scores = torch.zeros(2, 256, device="cuda")
    tri.score(kv, c, w.theta, w.offsets, inp.p_cur, scores)
    torch.cuda.synchronize()
    assert int(kv.dev_status.item()) == tri.DEV_NVALID_OVER_CAP
    kv.dev_status.zero_()
    keep = torch.zeros(2, 128, dtype=torch.int32, device="cuda")
    tri.select_topk(scores, kv, 0, 0, 128, keep)
    torch.cuda.synchronize()
    assert int(kv.dev_status.item()) == tri.DEV_NVALID_OVER_CAP


@pytest.mark.parametrize("wname", ["tiny", "qwen3_8b_layer"])
def test_pipeline_against_oracle(wname):
    """calibrate -> score -> select -> compact on the GPU vs the oracle
    pipeline from the same queries and cache (near-tie rule on the keep
    sets, exact bytes for the compaction)."""
    w = synth.WORKLOADS[wname]
    inp = synth.make_inputs(w, "cuda")
    S, n_cap, P, W, B = w.n_slices, w.n_cap, w.n_prompt, w.n_recent, w.budget
    pristine = (inp.k.clone(), inp.v.clone())
    c = tri.calibrate_centers(inp.q, w.group)
    kv = make_cache(inp)
    scores = torch.zeros(S, n_cap, device="cuda")
    keep = torch.zeros(S, B, dtype=torch.int32, device="cuda")
    tri.score(kv, c, w.theta, w.offsets, inp.p_cur, scores, n_prompt=P, n_recent=W)
    tri.select_topk(scores, kv, P, W, B, keep)
    tri.compact_kv(kv, keep, B)
    torch.cuda.synchronize()
    assert int(kv.dev_status.item()) == 0
    rc = orc.calibrate(f64(inp.q), w.group)
    g_keep = keep.cpu().numpy()
    g_scores = scores.cpu().numpy()
    total_swaps = 0
    for s in range(S):
        n = w.n_valid
        seq, lh = seq_lh(inp, s)
        k_np = f64(slice_rows(pristine[0], s)[:n])
        sref = orc.score_series(k_np, rc[0][lh], rc[1][lh], rc[2][lh], w.offsets, int(inp.p_cur[seq]), w.theta)
        M = orc.score_bound(k_np, rc[1][lh])
        problems, swaps = near_tie_violations(g_keep[s], sref, M, n, P, W, B)
        assert not problems, (s, problems)
        total_swaps += swaps
        # same precision decides the same set: oracle selection on the GPU's fp32 scores
        sc = g_scores[s].astype(np.float64)
        assert np.array_equal(g_keep[s], orc.select(sc, n, P, W, B))
        for cur, pr in ((kv.k, pristine[0]), (kv.v, pristine[1])):
            rows = slice_rows(pr, s).cpu().contiguous().view(torch.uint8).numpy().reshape(n_cap, -1).copy()
            orc.compact(rows, g_keep[s])
            got = slice_rows(cur, s).cpu().contiguous().view(torch.uint8).numpy().reshape(n_cap, -1)
            assert np.array_equal(got, rows)
        assert np.array_equal(kv.pos_out[s, :B].cpu().numpy(), g_keep[s])
    assert torch.all(kv.n_valid == B)
    print(f"{wname}: near-tie swaps vs oracle ranking: {total_swaps}")


@pytest.mark.parametrize("n_cap,P,W,B,nv", [
    (150001, 100, 10, 90000, [150001, 150000, 70000, 149999]),  # beyond one bitmap: exact fallback, pieces
    (5000, 7, 3, 4998, [5000, 5000, 4999, 4000]),                 # keep nearly all
    (300, 0, 0, 10, [300, 11, 10, 299]),                          # tiny candidate sets
])
def test_random_bit_exact_edge_shapes(n_cap, P, W, B, nv):
    k = torch.zeros(1, 2, 2, n_cap, 64, dtype=torch.bfloat16, device="cuda")
    kv = tri.KVCache(k, k, torch.tensor(nv, dtype=torch.int32, device="cuda"), None, None,
                     torch.zeros(1, dtype=torch.int32, device="cuda"))
    keep = torch.full((4, B), -9, dtype=torch.int32, device="cuda")
    tri.rand_evict(kv, 77, 3, P, W, B, keep)
    torch.cuda.synchronize()
    g = keep.cpu().numpy()
    for s in range(4):
        layer, head = divmod(s, 2)
        exp = orc.rand_select(77, 3, 0, layer, head, nv[s], P, W, B)
        assert np.array_equal(g[s], exp), s
    assert int(kv.dev_status.item()) == 0


def _compress_vs_separate(w, ragged=False, explicit_pos=False, seed=0, style=0):
    """tri_compress must equal tri_score + tri_select_topk + tri_compact_kv."""
    inp = synth.make_inputs(w, "cuda")
    S, n_cap, P, W, B = w.n_slices, w.n_cap, w.n_prompt, w.n_recent, w.budget
    rng = np.random.default_rng(seed)
    if ragged:
        nv = rng.integers(0, n_cap + 1, size=S)
        nv[0], nv[-1] = n_cap, B
        inp.n_valid = torch.tensor(nv, dtype=torch.int32, device="cuda")
    pos = None
    if explicit_pos:
        pos_np = np.stack([np.sort(rng.choice(3 * n_cap, size=n_cap, replace=False)) for _ in range(S)])
        pos = torch.tensor(pos_np, dtype=torch.int32, device="cuda")
        inp.p_cur = torch.full((w.n_seq,), 3 * n_cap + 1, dtype=torch.int64, device="cuda")
    c = tri.calibrate_centers(inp.q, w.group, style=style)
    k0, v0 = inp.k.clone(), inp.v.clone()
    # separate calls on a copy
    kv_a = tri.KVCache(k0.clone(), v0.clone(), inp.n_valid.clone(), None if pos is None else pos.clone(),
                       torch.zeros(S, n_cap, dtype=torch.int32, device="cuda"),
                       torch.zeros(1, dtype=torch.int32, device="cuda"))
    if pos is not None:
        kv_a.pos_out = kv_a.pos
    sc = torch.zeros(S, n_cap, device="cuda")
    keep_a = torch.full((S, B), -5, dtype=torch.int32, device="cuda")
    tri.score(kv_a, c, w.theta, w.offsets, inp.p_cur, sc, n_prompt=P, n_recent=W, style=style)
    tri.select_topk(sc, kv_a, P, W, B, keep_a)
    tri.compact_kv(kv_a, keep_a, B)
    # fused
    kv_b = tri.KVCache(k0.clone(), v0.clone(), inp.n_valid.clone(), None if pos is None else pos.clone(),
                       torch.zeros(S, n_cap, dtype=torch.int32, device="cuda"),
                       torch.zeros(1, dtype=torch.int32, device="cuda"))
    if pos is not None:
        kv_b.pos_out = kv_b.pos
    keep_b = torch.full((S, B), -5, dtype=torch.int32, device="cuda")
    ws = torch.empty(tri.compress_workspace_bytes(kv_b), dtype=torch.uint8, device="cuda")
    n0 = tri.launch_count()
    tri.compress(kv_b, c, w.theta, w.offsets, inp.p_cur, P, W, B, keep_b, workspace=ws, style=style)
    torch.cuda.synchronize()
    # a slice that fits one score CTA (32 tiles of 32 KB): score, selection and
    # compaction in one launch; else the three kernels
    tile_rows = 32768 // (w.head_dim * w.elem_bytes)
    rows_per_cta = min(32 * tile_rows, -(-n_cap // tile_rows) * tile_rows)
    assert tri.launch_count() - n0 == (1 if n_cap <= rows_per_cta else 3)
    # tri_select_compact on the separate call's scores: the same again
    kv_c = tri.KVCache(k0.clone(), v0.clone(), inp.n_valid.clone(), None if pos is None else pos.clone(),
                       torch.zeros(S, n_cap, dtype=torch.int32, device="cuda"),
                       torch.zeros(1, dtype=torch.int32, device="cuda"))
    if pos is not None:
        kv_c.pos_out = kv_c.pos
    keep_c = torch.full((S, B), -5, dtype=torch.int32, device="cuda")
    tri.select_compact(sc, kv_c, P, W, B, keep_c)
    torch.cuda.synchronize()
    for kv_x, keep_x in ((kv_b, keep_b), (kv_c, keep_c)):
        assert int(kv_a.dev_status.item()) == 0 and int(kv_x.dev_status.item()) == 0
        assert torch.equal(keep_a, keep_x)
        assert torch.equal(kv_a.k, kv_x.k) and torch.equal(kv_a.v, kv_x.v)
        assert torch.equal(kv_a.n_valid, kv_x.n_valid)
        nk = kv_a.n_valid.cpu().numpy()
        for s in range(S):
            assert torch.equal(kv_a.pos_out[s, :nk[s]], kv_x.pos_out[s, :nk[s]])
    # the scores left in the workspace are the separate call's scores
    fs = ws[: S * n_cap * 4].view(torch.float32).view(S, n_cap)
    nv_h = inp.n_valid.cpu().numpy()
    for s in range(S):
        lo, hi = P, int(nv_h[s]) - W
        if hi > lo:
            assert torch.equal(fs[s, lo:hi], sc[s, lo:hi])


@pytest.mark.parametrize("wname", ["tiny", "qwen3_8b_layer"])
def test_compress_equals_separate_calls(wname):
    _compress_vs_separate(synth.WORKLOADS[wname])


def test_compress_ragged_explicit_positions_and_styles():
    w = synth.scaled(LAYER, n_seq=2, n_layers=3, n_kv_heads=4, n_cap=5000, n_valid=5000, budget=1500,
                     n_prompt=100, n_recent=50, n_cal=512)
    _compress_vs_separate(w, ragged=True, seed=1)
    _compress_vs_separate(w, explicit_pos=True, seed=2, style=1)
    w2 = synth.scaled(TINY, dtype=torch.bfloat16, n_kv_heads=6, n_cap=3000, n_valid=3000, budget=700,
                      n_prompt=0, n_recent=0)
    _compress_vs_separate(w2, ragged=True, seed=3)
    w3 = synth.scaled(TINY, dtype=torch.bfloat16, n_kv_heads=5, n_cap=1001, n_valid=1001, budget=333,
                      n_prompt=3, n_recent=5)  # rows not a multiple of 4
    _compress_vs_separate(w3, ragged=True, seed=4)
