"""Paged caches (block tables per sequence; Random Attention, section 6: the
score is a pass through the block tables, eviction rewrites the survivors
into the request's blocks and frees the tail) through the C ABI.

The same rows laid out contiguously and through a shuffled block table must
give bit-identical scores, keep lists and compacted rows (the kernels differ
only in addressing); the contiguous path is itself checked against the
oracle elsewhere, and a few slices are checked against the oracle here too.
"""
import numpy as np
import pytest
import torch

import oracle as orc
import kv_cache_compression_tri_gb300 as tri
from kv_cache_compression_tri_gb300 import synth
from gpu_helpers import SCORE_TOL, f64, make_cache, seq_lh, slice_rows

pytestmark = pytest.mark.gpu

LAYER = synth.WORKLOADS["qwen3_8b_layer"]
TINY = synth.WORKLOADS["tiny"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    tri.load_library()


def _paged_copy(inp, bs, seed, spare=8, layout="blh"):
    """Pools holding the same logical rows as inp.k / inp.v, in blocks of bs
    rows scattered through a shuffled table. layout "blh": pools [nb][L][H][bs][d];
    "lbh": the layer outermost (a view with other strides). `spare` unused
    blocks are allocated past the ones the table may name."""
    n_seq, L, H, n_cap, d = inp.k.shape
    mb = n_cap // bs
    nb = n_seq * mb + 3  # a few blocks no table names
    rng = np.random.default_rng(seed)
    table = rng.permutation(nb)[: n_seq * mb].reshape(n_seq, mb).astype(np.int32)
    def pool():  # filled with noise, so a stray write would show
        if layout == "blh":
            return torch.randn(nb + spare, L, H, bs, d, device="cuda").to(inp.k.dtype)
        return torch.randn(L, nb + spare, H, bs, d, device="cuda").to(inp.k.dtype).permute(1, 0, 2, 3, 4)
    kp, vp = pool(), pool()
    t = torch.tensor(table, device="cuda", dtype=torch.long)
    for s in range(n_seq):
        ks = inp.k[s].reshape(L, H, mb, bs, d).permute(2, 0, 1, 3, 4)  # [mb][L][H][bs][d]
        vs = inp.v[s].reshape(L, H, mb, bs, d).permute(2, 0, 1, 3, 4)
        kp[t[s]] = ks
        vp[t[s]] = vs
    return kp[:nb], vp[:nb], torch.tensor(table, device="cuda"), kp, vp


def _logical(kp, table, s, n, L, H, bs):
    """Logical rows [0, n) of slice s of a paged pool, gathered on the host."""
    seq, rem = divmod(s, L * H)
    layer, head = divmod(rem, H)
    r = np.arange(n)
    blk = torch.tensor(np.asarray(table)[seq, r // bs], dtype=torch.long, device=kp.device)
    off = torch.tensor(r % bs, dtype=torch.long, device=kp.device)
    return kp[blk, layer, head, off]


@pytest.mark.parametrize("bs,layout", [(16, "blh"), (64, "lbh")])
def test_paged_score_select_compact_match_contiguous(bs, layout):
    w = synth.scaled(LAYER, n_seq=2, n_layers=2, n_kv_heads=4, n_cap=2176, n_valid=2176)
    inp = synth.make_inputs(w, "cuda")
    S, n_cap, L, H = w.n_slices, w.n_cap, w.n_layers, w.n_kv_heads
    P, W, B = w.n_prompt, w.n_recent, w.budget
    nv = np.full(S, n_cap)
    nv[1], nv[5] = 2000, 1500
    inp.n_valid = torch.tensor(nv, dtype=torch.int32, device="cuda")
    c = tri.calibrate_centers(inp.q, w.group)
    kp, vp, table, kp_full, vp_full = _paged_copy(inp, bs, seed=bs, layout=layout)
    pos = torch.tensor(np.stack([np.sort(np.random.default_rng(s).choice(3 * n_cap, n_cap, replace=False))
                                 for s in range(S)]), dtype=torch.int32, device="cuda")
    inp.p_cur = torch.full((w.n_seq,), 3 * n_cap + 1, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv_p = tri.PagedKVCache(kp, vp, table, inp.n_valid.clone(), pos.clone(), pos.clone(), st)
    kv_c = make_cache(inp, pos=pos.clone(), in_place_pos=True)
    sc_p = torch.full((S, n_cap), 5.0, device="cuda")
    sc_c = torch.full((S, n_cap), 5.0, device="cuda")
    tri.score(kv_p, c, w.theta, w.offsets, inp.p_cur, sc_p, n_prompt=P, n_recent=W)
    tri.score(kv_c, c, w.theta, w.offsets, inp.p_cur, sc_c, n_prompt=P, n_recent=W)
    torch.cuda.synchronize()
    assert torch.equal(sc_p, sc_c)
    # a few slices against the oracle directly
    cc, cm, cR = f64(c.center), f64(c.mean_norm), f64(c.mrl)
    tab = table.cpu().numpy()
    for s in (0, 5, S - 1):
        n = int(nv[s])
        seq, lh = seq_lh(inp, s)
        k = f64(_logical(kp, tab, s, n, L, H, bs))
        ref = orc.score_series(k, cc[lh], cm[lh], cR[lh], w.offsets, int(inp.p_cur[seq]), w.theta,
                               pos=pos[s, :n].cpu().numpy().astype(np.int64))
        M = orc.score_bound(k, cm[lh])
        assert np.all(np.abs(sc_p[s, P:n - W].cpu().numpy() - ref[P:n - W]) <= SCORE_TOL * M[P:n - W])
    # the fused selection + compaction on another paged copy must match the two calls below
    kp2, vp2, table2, _, _ = _paged_copy(inp, bs, seed=bs + 1, layout=layout)
    kv_f = tri.PagedKVCache(kp2, vp2, table2, inp.n_valid.clone(), pos.clone(), pos.clone(),
                            torch.zeros(1, dtype=torch.int32, device="cuda"))
    keep_f = torch.empty(S, B, dtype=torch.int32, device="cuda")
    tri.select_compact(sc_p, kv_f, P, W, B, keep_f)
    keep = torch.empty(S, B, dtype=torch.int32, device="cuda")
    tri.select_topk(sc_p, kv_p, P, W, B, keep)
    before = {s: _logical(kp, tab, s, int(nv[s]), L, H, bs).cpu() for s in range(S)}
    before_v = {s: _logical(vp, tab, s, int(nv[s]), L, H, bs).cpu() for s in range(S)}
    untouched = kp_full[kp.shape[0]:].clone(), vp_full[kp.shape[0]:].clone()
    tri.compact_kv(kv_p, keep, B)
    tri.compact_kv(kv_c, keep, B)
    used = torch.empty(w.n_seq, dtype=torch.int32, device="cuda")
    tri.paged_blocks_used(kv_p, used)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(kv_p.n_valid, kv_c.n_valid) and torch.equal(kv_p.pos_out, kv_c.pos_out)
    g_keep = keep.cpu().numpy()
    for s in range(S):
        n_keep = int(kv_p.n_valid[s])
        k_after = _logical(kp, tab, s, n_keep, L, H, bs).cpu()
        assert torch.equal(k_after, slice_rows(kv_c.k, s)[:n_keep].cpu())
        assert torch.equal(_logical(vp, tab, s, n_keep, L, H, bs).cpu(), slice_rows(kv_c.v, s)[:n_keep].cpu())
        # the oracle's in-place byte loop on the logical rows gives the same
        rows = before[s].view(torch.int16).numpy().copy()
        orc.compact(rows, g_keep[s])
        assert np.array_equal(rows[:n_keep], k_after.view(torch.int16).numpy())
        rows_v = before_v[s].view(torch.int16).numpy().copy()
        orc.compact(rows_v, g_keep[s])
        assert np.array_equal(rows_v[:n_keep], _logical(vp, tab, s, n_keep, L, H, bs).cpu().view(torch.int16).numpy())
    assert torch.equal(keep_f, keep) and torch.equal(kv_f.n_valid, kv_p.n_valid)
    tab2 = table2.cpu().numpy()
    for s in range(S):
        n_keep = int(kv_p.n_valid[s])
        assert torch.equal(_logical(kp2, tab2, s, n_keep, L, H, bs), _logical(kp, tab, s, n_keep, L, H, bs))
        assert torch.equal(_logical(vp2, tab2, s, n_keep, L, H, bs), _logical(vp, tab, s, n_keep, L, H, bs))
    # blocks past the table's reach were not written; the tail is free
    assert torch.equal(kp_full[kp.shape[0]:], untouched[0]) and torch.equal(vp_full[kp.shape[0]:], untouched[1])
    assert used.cpu().tolist() == [(B + bs - 1) // bs] * w.n_seq


def test_paged_gqa_compress_and_post_rope():
    w = synth.scaled(LAYER, n_kv_heads=2, n_layers=2, n_cap=1024, n_valid=1024, n_cal=512, n_prompt=64,
                     n_recent=32, budget=300)
    inp = synth.make_inputs(w, "cuda")
    S, n_cap, G = w.n_slices, w.n_cap, w.group
    kp, vp, table, _, _ = _paged_copy(inp, 32, seed=3)
    # GQA scores and statistics: identical to the contiguous layout
    cq = tri.calibrate_centers(inp.q, 1)
    kv_p = tri.PagedKVCache(kp, vp, table, inp.n_valid.clone(), None, torch.empty(S, n_cap, dtype=torch.int32,
                                                                                   device="cuda"),
                            torch.zeros(1, dtype=torch.int32, device="cuda"))
    kv_c = make_cache(inp)
    out = []
    for kv in (kv_p, kv_c):
        sg = torch.empty(S, G, n_cap, device="cuda")
        stt = torch.empty(S, G, 2, device="cuda")
        tri.score_heads(kv, cq, G, w.theta, w.offsets, inp.p_cur, sg, stt)
        out.append((sg, stt))
    torch.cuda.synchronize()
    assert torch.equal(out[0][0], out[1][0]) and torch.equal(out[0][1], out[1][1])
    # one tri_compress call: the same keep lists and rows as contiguous
    c = tri.calibrate_centers(inp.q, w.group)
    kp2, vp2, table2, _, _ = _paged_copy(inp, 32, seed=4)
    kv_p = tri.PagedKVCache(kp2, vp2, table2, inp.n_valid.clone(), None,
                            torch.empty(S, n_cap, dtype=torch.int32, device="cuda"),
                            torch.zeros(1, dtype=torch.int32, device="cuda"))
    kv_c = make_cache(inp)
    keeps = []
    for kv in (kv_p, kv_c):
        keep = torch.empty(S, w.budget, dtype=torch.int32, device="cuda")
        tri.compress(kv, c, w.theta, w.offsets, inp.p_cur, w.n_prompt, w.n_recent, w.budget, keep)
        keeps.append(keep)
    torch.cuda.synchronize()
    assert torch.equal(keeps[0], keeps[1])
    tab = table2.cpu().numpy()
    for s in range(S):
        assert torch.equal(_logical(kp2, tab, s, w.budget, w.n_layers, w.n_kv_heads, 32).cpu(),
                           slice_rows(kv_c.k, s)[:w.budget].cpu())
    # post-RoPE keys in a paged pool score like the same keys contiguous
    wp = synth.scaled(w, key_layout="post")
    inp2 = synth.make_inputs(wp, "cuda")
    kp3, vp3, table3, _, _ = _paged_copy(inp2, 16, seed=5)
    kv_p = tri.PagedKVCache(kp3, vp3, table3, inp2.n_valid.clone(), None, None, post_rope=True)
    kv_c = make_cache(inp2)
    kv_c.post_rope = True
    scs = []
    for kv in (kv_p, kv_c):
        sc = torch.empty(S, n_cap, device="cuda")
        tri.score(kv, c, wp.theta, wp.offsets, inp2.p_cur, sc)
        scs.append(sc)
    torch.cuda.synchronize()
    assert torch.equal(scs[0], scs[1])


def test_paged_compaction_past_the_shared_table_copy():
    """A compaction CTA keeps the table entries of 2000 blocks (from the block
    of the first row that moves) in shared memory and reads later ones from
    the table: 32768-row slices in 16-row blocks with nothing protected use
    both, through the standalone compaction and the fused random
    selection + compaction."""
    w = synth.scaled(LAYER, n_seq=1, n_layers=1, n_kv_heads=2, n_cap=32768, n_valid=32768, budget=4096,
                     n_prompt=0, n_recent=64, n_cal=256)
    inp = synth.make_inputs(w, "cuda")
    S, n_cap, L, H, B, W, bs = w.n_slices, w.n_cap, w.n_layers, w.n_kv_heads, w.budget, w.n_recent, 16
    assert n_cap // bs > 2000
    c = tri.calibrate_centers(inp.q, w.group)
    sc = torch.empty(S, n_cap, device="cuda")
    tri.score(make_cache(inp), c, w.theta, w.offsets, inp.p_cur, sc, n_prompt=0, n_recent=W)
    keep = torch.empty(S, B, dtype=torch.int32, device="cuda")
    tri.select_topk(sc, make_cache(inp), 0, W, B, keep)
    torch.cuda.synchronize()
    before_k = [slice_rows(inp.k, s).clone() for s in range(S)]
    keep_h = keep.cpu().numpy()
    assert keep_h[:, 0].max() < 2000 * bs and keep_h[:, -1].min() >= 2000 * bs  # both halves of the table
    for fused in (False, True):
        kp, vp, table, _, _ = _paged_copy(inp, bs, seed=11 + fused)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        kv_p = tri.PagedKVCache(kp, vp, table, inp.n_valid.clone(), None,
                                torch.empty(S, n_cap, dtype=torch.int32, device="cuda"), st)
        kv_c = tri.KVCache(inp.k.clone(), inp.v.clone(), inp.n_valid.clone(), None,
                           torch.empty(S, n_cap, dtype=torch.int32, device="cuda"),
                           torch.zeros(1, dtype=torch.int32, device="cuda"))
        if fused:
            kps, kcs = torch.empty_like(keep), torch.empty_like(keep)
            tri.rand_evict_compact(kv_p, 5, 1, 0, W, B, kps)
            tri.rand_evict_compact(kv_c, 5, 1, 0, W, B, kcs)
        else:
            kps = kcs = keep
            tri.compact_kv(kv_p, keep, B)
            tri.compact_kv(kv_c, keep, B)
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and int(kv_c.dev_status.item()) == 0
        assert torch.equal(kps, kcs) and torch.equal(kv_p.n_valid, kv_c.n_valid)
        tab = table.cpu().numpy()
        for s in range(S):
            assert torch.equal(_logical(kp, tab, s, B, L, H, bs), slice_rows(kv_c.k, s)[:B]), (fused, s)
            assert torch.equal(_logical(vp, tab, s, B, L, H, bs), slice_rows(kv_c.v, s)[:B]), (fused, s)
            assert torch.equal(kv_p.pos_out[s, :B], kv_c.pos_out[s, :B])
        # the oracle's in-place byte loop on the logical rows gives the same
        rows = before_k[0].cpu().view(torch.int16).numpy().copy()
        orc.compact(rows, kps[0].cpu().numpy())
        assert np.array_equal(rows[:B], _logical(kp, tab, 0, B, L, H, bs).cpu().view(torch.int16).numpy())


def test_paged_bad_block_entry_sets_status():
    # the bad entry names a block that is allocated (a spare past num_blocks),
    # so nothing can leave the pool even if the check were missing
    w = synth.scaled(LAYER, n_kv_heads=2, n_cap=512, n_valid=512, n_cal=256, n_prompt=16, n_recent=16, budget=100)
    inp = synth.make_inputs(w, "cuda")
    S = w.n_slices
    kp, vp, table, kp_full, vp_full = _paged_copy(inp, 16, seed=6, spare=8)
    nb = kp.shape[0]
    table[0, 7] = nb + 3
    c = tri.calibrate_centers(inp.q, w.group)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # the pool handed over is the first nb blocks; the spares behind it are allocated
    kv = tri.PagedKVCache(kp_full[:nb], vp_full[:nb], table, inp.n_valid.clone(), None,
                          torch.empty(S, 512, dtype=torch.int32, device="cuda"), st)
    assert kv._abi().num_blocks == nb and kp_full.shape[0] == nb + 8
    sc = torch.zeros(S, 512, device="cuda")
    tri.score(kv, c, w.theta, w.offsets, inp.p_cur, sc)
    torch.cuda.synchronize()
    assert int(st.item()) == tri.DEV_BAD_BLOCK
    st.zero_()
    keep = torch.arange(100, 200, dtype=torch.int32, device="cuda").repeat(S, 1)
    spare_before = kp_full[nb:].clone()
    tri.compact_kv(kv, keep, 100)
    torch.cuda.synchronize()
    assert int(st.item()) == tri.DEV_BAD_BLOCK
    assert torch.equal(kp_full[nb:], spare_before)
