"""GPU parity at full size, in the launch configuration bench.py times.

  * qwen3_8b_stack  (16 x 36 x 8 slices, 32768 rows, d 128): every slice's
    keep list passes the structural invariants; 48 sampled slices are
    compared with the oracle (scores within tolerance, near-tie rule, exact
    selection on the same fp32 scores, exact compaction bytes).
  * random_stack    (same shapes, Random Attention): every slice's keep list
    equals the oracle's bit for bit; sampled slices' compaction bytes match.
  * periodic_large_batch (64 x 24 x 8 slices, d 64): the 32768-row event and
    16 periodic rounds of +128 rows with explicit positions; sampled slices
    are tracked by the oracle through every round.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import kv_cache_compression_tri_gb300 as tri
from kv_cache_compression_tri_gb300 import synth
from gpu_helpers import (CALIB_TOL, SCORE_TOL, f64, near_tie_violations, pmap, seq_lh, slice_rows)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    tri.load_library()
    yield
    torch.cuda.empty_cache()


def _rows_bytes(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).numpy().reshape(t.shape[0], -1)


def _structural(keep_all: np.ndarray, n: int, P: int, W: int, B: int):
    # every slice: ascending, in range, protected rows present, exactly B kept
    assert keep_all.shape[1] == B
    assert np.all(np.diff(keep_all, axis=1) > 0)
    assert np.all(keep_all[:, :P] == np.arange(P)[None, :])
    if W:
        assert np.all(keep_all[:, B - W:] == np.arange(n - W, n)[None, :])
    assert keep_all.min() >= 0 and keep_all.max() < n


def test_qwen3_stack_full_size():
    w = synth.WORKLOADS["qwen3_8b_stack"]
    S, n_cap, n, P, W, B, d = w.n_slices, w.n_cap, w.n_valid, w.n_prompt, w.n_recent, w.budget, w.head_dim
    inp = synth.make_inputs(w, "cuda")
    c = tri.calibrate_centers(inp.q, w.group)
    torch.cuda.synchronize()
    sample = synth.sample_slices(S, 48)
    # calibration parity on the (layer, head)s of the sampled slices
    lhs = sorted({seq_lh(inp, s)[1] for s in sample})
    gc, gm, gR = f64(c.center), f64(c.mean_norm), f64(c.mrl)
    for lh in lhs[:12]:
        layer, h = divmod(lh, w.n_kv_heads)
        q = f64(inp.q[layer, h * w.group:(h + 1) * w.group])[None]
        rc, rm, rR = orc.calibrate(q, w.group)
        assert np.all(np.abs(gc[lh] - rc[0]) <= CALIB_TOL * rm[0][:, None])
        assert np.all(np.abs(gm[lh] - rm[0]) <= CALIB_TOL * rm[0])
        assert np.all(np.abs(gR[lh] - rR[0]) <= CALIB_TOL)
    inp.q = None
    torch.cuda.empty_cache()

    pk = {s: slice_rows(inp.k, s).cpu() for s in sample}
    pv = {s: slice_rows(inp.v, s).cpu() for s in sample}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos_out = torch.empty(S, n_cap, dtype=torch.int32, device="cuda")
    kv = tri.KVCache(inp.k, inp.v, inp.n_valid.clone(), None, pos_out, status)
    scores = torch.empty(S, n_cap, device="cuda")
    keep = torch.empty(S, B, dtype=torch.int32, device="cuda")
    tri.score(kv, c, w.theta, w.offsets, inp.p_cur, scores, n_prompt=P, n_recent=W)
    tri.select_topk(scores, kv, P, W, B, keep)
    tri.compact_kv(kv, keep, B)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    keep_all = keep.cpu().numpy()
    _structural(keep_all, n, P, W, B)
    assert torch.all(kv.n_valid == B)
    assert torch.equal(pos_out[:, :B], keep)
    g_scores = {s: scores[s].cpu().numpy() for s in sample}
    g_k = {s: slice_rows(inp.k, s)[:B].cpu() for s in sample}
    g_v = {s: slice_rows(inp.v, s)[:B].cpu() for s in sample}

    def check(s):
        seq, lh = seq_lh(inp, s)
        k64 = pk[s].to(torch.float64).numpy()
        sref = np.full(n, np.nan)
        sref[P:n - W] = orc.score_series(k64[P:n - W], gc[lh], gm[lh], gR[lh], w.offsets, int(inp.p_cur[seq]),
                                         w.theta, pos=np.arange(P, n - W))
        M = orc.score_bound(k64, gm[lh])
        err = np.abs(g_scores[s][P:n - W] - sref[P:n - W]) / M[P:n - W]
        full = np.where(np.isnan(sref), 0.0, sref)
        problems, swaps = near_tie_violations(keep_all[s], full, M, n, P, W, B)
        exact = np.array_equal(keep_all[s], orc.select(g_scores[s].astype(np.float64), n, P, W, B))
        kb, vb = _rows_bytes(pk[s]).copy(), _rows_bytes(pv[s]).copy()
        orc.compact(kb, keep_all[s])
        orc.compact(vb, keep_all[s])
        same = np.array_equal(_rows_bytes(g_k[s]), kb[:B]) and np.array_equal(_rows_bytes(g_v[s]), vb[:B])
        return float(err.max()), problems, swaps, exact, same

    res = pmap(check, sample)
    worst = max(r[0] for r in res)
    assert worst <= SCORE_TOL, worst
    for s, r in zip(sample, res):
        assert not r[1], (s, r[1])
        assert r[3], f"slice {s}: selection differs from the oracle on identical fp32 scores"
        assert r[4], f"slice {s}: compacted bytes differ"
    print(f"qwen3_8b_stack: worst score error/M {worst:.2e}, near-tie swaps {sum(r[2] for r in res)}")


def test_random_stack_full_size():
    w = synth.WORKLOADS["random_stack"]
    S, n_cap, n, P, W, B = w.n_slices, w.n_cap, w.n_valid, w.n_prompt, w.n_recent, w.budget
    inp = synth.make_inputs(w, "cuda", with_queries=False)
    sample = synth.sample_slices(S, 16)
    pk = {s: slice_rows(inp.k, s).cpu() for s in sample}
    pv = {s: slice_rows(inp.v, s).cpu() for s in sample}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos_out = torch.empty(S, n_cap, dtype=torch.int32, device="cuda")
    kv = tri.KVCache(inp.k, inp.v, inp.n_valid.clone(), None, pos_out, status)
    keep = torch.empty(S, B, dtype=torch.int32, device="cuda")
    tri.rand_evict(kv, 0, 0, P, W, B, keep)
    tri.compact_kv(kv, keep, B)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    keep_all = keep.cpu().numpy()
    L, H = w.n_layers, w.n_kv_heads

    def ref(s):
        seq, rem = divmod(s, L * H)
        layer, head = divmod(rem, H)
        return np.array_equal(keep_all[s], orc.rand_select(0, 0, seq, layer, head, n, P, W, B))

    ok = pmap(ref, range(S))
    assert all(ok), f"{ok.count(False)} slices differ"
    for s in sample:
        kb, vb = _rows_bytes(pk[s]).copy(), _rows_bytes(pv[s]).copy()
        orc.compact(kb, keep_all[s])
        orc.compact(vb, keep_all[s])
        assert np.array_equal(_rows_bytes(slice_rows(inp.k, s)[:B].cpu()), kb[:B])
        assert np.array_equal(_rows_bytes(slice_rows(inp.v, s)[:B].cpu()), vb[:B])
    assert torch.all(kv.n_valid == B)


@pytest.mark.parametrize("view", ["full_capacity", "steady_state"])
def test_periodic_large_batch_full_size(view):
    """Rounds run either on the whole 32768-row capacity (n_valid << n_cap)
    or, as an engine would in steady state, on a view of capacity B + 128
    (same storage and slice stride)."""
    w = synth.WORKLOADS["periodic_large_batch"]
    S, n_cap, P, W, B, d = w.n_slices, w.n_cap, w.n_prompt, w.n_recent, w.budget, w.head_dim
    R = w.round_rows
    inp = synth.make_inputs(w, "cuda")
    c = tri.calibrate_centers(inp.q, w.group)
    inp.q = None
    torch.cuda.synchronize()
    gc, gm, gR = f64(c.center), f64(c.mean_norm), f64(c.mrl)
    sample = synth.sample_slices(S, 24)
    # oracle-side state of the sampled slices: key rows (fp64 and bytes), value bytes, positions
    st = {s: {"k": slice_rows(inp.k, s).cpu().clone(), "v": slice_rows(inp.v, s).cpu().clone(),
              "pos": np.arange(n_cap, dtype=np.int64), "n": w.n_valid} for s in sample}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.empty(S, n_cap, dtype=torch.int32, device="cuda")
    kv = tri.KVCache(inp.k, inp.v, inp.n_valid.clone(), None, pos, status)
    scores = torch.empty(S, n_cap, device="cuda")
    keep = torch.empty(S, B, dtype=torch.int32, device="cuda")
    p_cur = inp.p_cur.clone()
    total_swaps, worst = 0, 0.0
    for rnd in range(w.rounds + 1):
        if rnd == 1 and view == "steady_state":
            cap = B + R
            pos = pos[:, :cap].clone()
            kv = tri.KVCache(inp.k[:, :, :, :cap], inp.v[:, :, :, :cap], kv.n_valid, pos, pos, status)
            # the bench's rounds: one tri_compress call, each slice scored,
            # selected and compacted by one CTA (scores left in the workspace)
            cws = torch.empty(tri.compress_workspace_bytes(kv), dtype=torch.uint8, device="cuda")
            scores = cws[: S * cap * 4].view(torch.float32).view(S, cap)
        if rnd > 0:
            kn, vn = synth.append_rows(inp, rnd, R)
            inp.k[:, :, :, B:B + R] = kn
            inp.v[:, :, :, B:B + R] = vn
            first = n_cap + R * (rnd - 1)
            pos[:, B:B + R] = torch.arange(first, first + R, dtype=torch.int32, device="cuda")[None, :]
            kv.n_valid.fill_(B + R)
            p_cur.fill_(first + R - 1)
            kv.pos = pos  # positions are explicit after the first compaction (in place)
            knh = kn.view(S, R, d)
            vnh = vn.view(S, R, d)
            for s in sample:
                st[s]["k"][B:B + R] = knh[s].cpu()
                st[s]["v"][B:B + R] = vnh[s].cpu()
                st[s]["pos"][B:B + R] = np.arange(first, first + R)
                st[s]["n"] = B + R
        if view == "steady_state" and rnd > 0:
            n0 = tri.launch_count()
            tri.compress(kv, c, w.theta, w.offsets, p_cur, P, W, B, keep, workspace=cws)
            assert tri.launch_count() - n0 == 1
        else:
            tri.score(kv, c, w.theta, w.offsets, p_cur, scores, n_prompt=P, n_recent=W)
            tri.select_topk(scores, kv, P, W, B, keep)
            tri.compact_kv(kv, keep, B)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, rnd
        keep_all = keep.cpu().numpy()
        n_now = w.n_valid if rnd == 0 else B + R
        _structural(keep_all, n_now, P, W, B)
        pc = int(p_cur[0])
        gs = {s: scores[s, :n_now].cpu().numpy() for s in sample}

        def check(s):
            x = st[s]
            n = x["n"]
            seq, lh = seq_lh(inp, s)
            k64 = x["k"][:n].to(torch.float64).numpy()
            sref = orc.score_series(k64, gc[lh], gm[lh], gR[lh], w.offsets, pc, w.theta, pos=x["pos"][:n])
            M = orc.score_bound(k64, gm[lh])
            err = np.abs(gs[s][P:n - W] - sref[P:n - W]) / M[P:n - W]
            problems, swaps = near_tie_violations(keep_all[s], sref, M, n, P, W, B)
            sc = gs[s].astype(np.float64)
            sc[:P] = 0.0  # rows outside the candidates are not scored (the fused call leaves them as they were)
            sc[n - W:] = 0.0
            exact = np.array_equal(keep_all[s], orc.select(sc, n, P, W, B))
            return float(err.max()), problems, swaps, exact

        res = pmap(check, sample)
        for s, r in zip(sample, res):
            assert r[0] <= SCORE_TOL, (rnd, s, r[0])
            assert not r[1], (rnd, s, r[1])
            assert r[3], (rnd, s)
            worst = max(worst, r[0])
            total_swaps += r[2]
        # advance the oracle state with the GPU keep lists and compare bytes and positions
        for s in sample:
            x = st[s]
            kb, vb = _rows_bytes(x["k"]).copy(), _rows_bytes(x["v"]).copy()
            orc.compact(kb, keep_all[s])
            orc.compact(vb, keep_all[s])
            x["k"] = torch.from_numpy(kb.copy()).view(torch.bfloat16).view(n_cap, d)
            x["v"] = torch.from_numpy(vb.copy()).view(torch.bfloat16).view(n_cap, d)
            x["pos"][:B] = x["pos"][keep_all[s]]
            x["n"] = B
            assert np.array_equal(_rows_bytes(slice_rows(inp.k, s)[:B].cpu()), kb[:B]), (rnd, s)
            assert np.array_equal(_rows_bytes(slice_rows(inp.v, s)[:B].cpu()), vb[:B]), (rnd, s)
            assert np.array_equal(pos[s, :B].cpu().numpy(), x["pos"][:B]), (rnd, s)
        assert torch.all(kv.n_valid == B)
    print(f"periodic: worst score error/M {worst:.2e}, near-tie swaps {total_swaps} over {w.rounds + 1} events")


def test_qwen3_stack_full_size_compress():
    """The single-call entry point at full size: keep lists follow the oracle on
    sampled slices (exactly, on the fp32 scores it left in its workspace, and
    by the near-tie rule against fp64 scores) and the structural invariants
    hold for every slice."""
    w = synth.WORKLOADS["qwen3_8b_stack"]
    S, n_cap, n, P, W, B = w.n_slices, w.n_cap, w.n_valid, w.n_prompt, w.n_recent, w.budget
    inp = synth.make_inputs(w, "cuda")
    c = tri.calibrate_centers(inp.q, w.group)
    inp.q = None
    sample = synth.sample_slices(S, 24)
    pk = {s: slice_rows(inp.k, s).cpu() for s in sample}
    pv = {s: slice_rows(inp.v, s).cpu() for s in sample}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv = tri.KVCache(inp.k, inp.v, inp.n_valid.clone(), None,
                     torch.empty(S, n_cap, dtype=torch.int32, device="cuda"), status)
    keep = torch.empty(S, B, dtype=torch.int32, device="cuda")
    ws = torch.empty(tri.compress_workspace_bytes(kv), dtype=torch.uint8, device="cuda")
    tri.compress(kv, c, w.theta, w.offsets, inp.p_cur, P, W, B, keep, workspace=ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    keep_all = keep.cpu().numpy()
    _structural(keep_all, n, P, W, B)
    assert torch.all(kv.n_valid == B)
    fs = ws[: S * n_cap * 4].view(torch.float32).view(S, n_cap)
    gc, gm, gR = f64(c.center), f64(c.mean_norm), f64(c.mrl)
    gs = {s: fs[s].cpu().numpy() for s in sample}

    def check(s):
        seq, lh = seq_lh(inp, s)
        k64 = pk[s].to(torch.float64).numpy()
        sref = np.zeros(n)
        sref[P:n - W] = orc.score_series(k64[P:n - W], gc[lh], gm[lh], gR[lh], w.offsets, int(inp.p_cur[seq]),
                                         w.theta, pos=np.arange(P, n - W))
        M = orc.score_bound(k64, gm[lh])
        err = float((np.abs(gs[s][P:n - W] - sref[P:n - W]) / M[P:n - W]).max())
        problems, _ = near_tie_violations(keep_all[s], sref, M, n, P, W, B)
        sc = gs[s].astype(np.float64)
        sc[:P] = 0.0
        sc[n - W:] = 0.0
        exact = np.array_equal(keep_all[s], orc.select(sc, n, P, W, B))
        kb, vb = _rows_bytes(pk[s]).copy(), _rows_bytes(pv[s]).copy()
        orc.compact(kb, keep_all[s])
        orc.compact(vb, keep_all[s])
        same = (np.array_equal(_rows_bytes(slice_rows(inp.k, s)[:B].cpu()), kb[:B])
                and np.array_equal(_rows_bytes(slice_rows(inp.v, s)[:B].cpu()), vb[:B]))
        return err, problems, exact, same

    res = pmap(check, sample)
    for s, r in zip(sample, res):
        assert r[0] <= SCORE_TOL, (s, r[0])
        assert not r[1], (s, r[1])
        assert r[2], s
        assert r[3], s
