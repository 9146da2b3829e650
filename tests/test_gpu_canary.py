"""Canary checks in place of a device memory checker (none is available to
these tests): every buffer an entry point is handed sits between guard
bytes, each cache slice is followed by guard rows (a slice stride larger
than n_cap rows), and everything an entry point must leave alone is
compared byte for byte with its state before the call:

  * the guard bytes before and after every buffer, and the guard rows past
    n_cap in every slice of K and V;
  * inputs (queries, centres, scores read by a selection, positions);
  * K, V and position rows at or past a slice's kept count (the compaction
    writes rows j < n_keep only, n_keep = min(n_valid, budget));
  * score rows outside the rows a call scores ([P, n - W) for tri_score and
    tri_compress, [0, n) for the per-head and union paths);
  * workspace bytes past the size the call asked for.

Ragged row counts cover 0, 1, the budget, one over it, rows not a multiple
of 4, and n_valid = n_cap."""
import numpy as np
import pytest
import torch

import kv_cache_compression_tri_gb300 as tri
from kv_cache_compression_tri_gb300 import synth

pytestmark = pytest.mark.gpu

SENT = 0xA5
PAD = 256  # guard bytes on each side of a buffer (keeps 16-byte alignment)
GAP = 8    # guard rows after each cache slice
_INT = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    tri.load_library()


class Guarded:
    """A tensor of `shape` inside a byte buffer with PAD guard bytes on each
    side, all filled with SENT before `init` (if given) is copied in."""

    def __init__(self, shape, dtype, init=None):
        self.shape, self.dtype = tuple(shape), dtype
        self.n = int(np.prod(self.shape)) * torch.tensor([], dtype=dtype).element_size()
        self.buf = torch.full((PAD + self.n + PAD,), SENT, dtype=torch.uint8, device="cuda")
        self.t = self.buf[PAD:PAD + self.n].view(dtype).view(self.shape)
        if init is not None:
            self.t.copy_(init)
        self.snap()

    def snap(self):
        self.before = self.buf.clone()

    def raw(self, b):
        return b[PAD:PAD + self.n].view(self.dtype).view(self.shape).view(_INT[self.t.element_size()])

    def check(self, allowed=None, what=""):
        """Guards intact and nothing outside `allowed` (a bool mask of shape,
        True where the call may write; None: nothing) changed."""
        torch.cuda.synchronize()
        assert torch.equal(self.buf[:PAD], self.before[:PAD]), f"{what}: guard before the buffer written"
        assert torch.equal(self.buf[PAD + self.n:], self.before[PAD + self.n:]), f"{what}: guard after the buffer written"
        a, b = self.raw(self.buf), self.raw(self.before)
        if allowed is None:
            assert torch.equal(a, b), f"{what}: written"
        else:
            keep = ~allowed
            assert torch.equal(a[keep], b[keep]), f"{what}: written outside the allowed region"


class GuardedCache:
    """K, V [n_seq, L, H, n_cap + GAP, d] guarded buffers; the cache is the
    view of the first n_cap rows of each slice."""

    def __init__(self, k, v, n_valid, pos=None, pos_out=True, post_rope=False):
        n_seq, L, H, n_cap, d = k.shape
        self.S, self.n_cap, self.d = n_seq * L * H, n_cap, d
        full = (n_seq, L, H, n_cap + GAP, d)
        self.gk, self.gv = Guarded(full, k.dtype), Guarded(full, k.dtype)
        self.gk.t[:, :, :, :n_cap].copy_(k)
        self.gv.t[:, :, :, :n_cap].copy_(v)
        self.gn = Guarded((self.S,), torch.int32, n_valid)
        self.gst = Guarded((1,), torch.int32, torch.zeros(1, dtype=torch.int32))
        self.gpos = Guarded((self.S, n_cap), torch.int32, pos) if pos is not None else None
        self.gpo = Guarded((self.S, n_cap), torch.int32, torch.full((self.S, n_cap), -3, dtype=torch.int32)) \
            if pos_out else None
        self.kv = tri.KVCache(self.gk.t[:, :, :, :n_cap], self.gv.t[:, :, :, :n_cap], self.gn.t,
                              self.gpos.t if self.gpos is not None else None,
                              self.gpo.t if self.gpo is not None else None, self.gst.t, post_rope=post_rope)
        self.nv0 = n_valid.cpu().numpy().copy()
        self.parts = [self.gk, self.gv, self.gn, self.gst] + [g for g in (self.gpos, self.gpo) if g is not None]
        self.snap()

    def snap(self):
        for g in self.parts:
            g.snap()

    def row_mask(self, n_rows: np.ndarray, width=None):
        """[S, n_cap(+GAP)] bool: rows j < n_rows[s] of each slice."""
        cols = self.n_cap + (GAP if width is None else 0)
        j = torch.arange(cols, device="cuda")[None, :]
        return j < torch.as_tensor(n_rows, device="cuda")[:, None]

    def check_untouched(self, what):
        for g in self.parts:
            allowed = None
            if g is self.gst:
                continue
            g.check(allowed, what)
        assert int(self.gst.t.item()) == 0, f"{what}: device status {int(self.gst.t.item())}"

    def check_compacted(self, B, what):
        n_keep = np.minimum(self.nv0, B)
        rows = self.row_mask(n_keep)  # [S, n_cap + GAP]
        n_seq, L, H = self.gk.shape[:3]
        kv_mask = rows.view(n_seq, L, H, self.n_cap + GAP, 1).expand(*self.gk.shape)
        self.gk.check(kv_mask, f"{what} K")
        self.gv.check(kv_mask, f"{what} V")
        self.gn.check(torch.ones(self.S, dtype=torch.bool, device="cuda"), f"{what} n_valid")
        if self.gpo is not None:
            self.gpo.check(self.row_mask(n_keep, width=0), f"{what} pos_out")
        if self.gpos is not None and self.gpos is not self.gpo:
            self.gpos.check(None, f"{what} pos")
        assert int(self.gst.t.item()) == 0, f"{what}: device status {int(self.gst.t.item())}"
        assert np.array_equal(self.gn.t.cpu().numpy(), n_keep), what


def _ragged(S, n_cap, B, seed):
    rng = np.random.default_rng(seed)
    nv = rng.integers(0, n_cap + 1, size=S)
    fixed = [0, 1, B, B + 1, n_cap, n_cap - 1, B + 3, 2 * B + 1][:S]
    nv[:len(fixed)] = [min(x, n_cap) for x in fixed]
    return torch.tensor(nv, dtype=torch.int32)


CASES = {
    # bf16, d 128, several score CTAs per slice (n_cap > 2048 rows), rows not a multiple of 4
    "bf16_d128": synth.scaled(synth.WORKLOADS["qwen3_8b_layer"], n_seq=2, n_layers=2, n_kv_heads=4, n_cap=4101,
                              n_valid=4101, budget=700, n_prompt=24, n_recent=16, n_cal=256),
    # fp32, d 64, one score CTA per slice (tri_compress's single-kernel path)
    "f32_d64": synth.scaled(synth.WORKLOADS["tiny"], n_seq=2, n_layers=2, n_kv_heads=4, n_cap=999, n_valid=999,
                            budget=301, n_prompt=8, n_recent=12, n_cal=256),
}


def _setup(name, seed=0, pos=False):
    w = CASES[name]
    inp = synth.make_inputs(w, "cuda")
    S, n_cap = w.n_slices, w.n_cap
    nv = _ragged(S, n_cap, w.budget, seed)
    p = None
    if pos:
        rng = np.random.default_rng(seed + 7)
        p = torch.tensor(np.stack([np.sort(rng.choice(3 * n_cap, size=n_cap, replace=False)) for _ in range(S)]),
                         dtype=torch.int32)
        inp.p_cur = torch.full((w.n_seq,), 3 * n_cap + 5, dtype=torch.int64, device="cuda")
    return w, inp, GuardedCache(inp.k, inp.v, nv, pos=p)


@pytest.mark.parametrize("name", list(CASES))
def test_canary_calibrate(name):
    w = CASES[name]
    inp = synth.make_inputs(w, "cuda")
    L, Hq, n_tok, d = inp.q.shape
    H, F = Hq // w.group, d // 2
    gq = Guarded(inp.q.shape, inp.q.dtype, inp.q)
    gc = Guarded((L * H, F, 2), torch.float32)
    gm = Guarded((L * H, F), torch.float32)
    gr = Guarded((L * H, F), torch.float32)
    need = tri.calibrate_workspace_bytes(L, Hq, w.group, d, n_tok)
    gw = Guarded((need,), torch.uint8)
    tri.calibrate_centers(gq.t, w.group, out=tri.Centers(gc.t, gm.t, gr.t), workspace=gw.t)
    gq.check(None, "queries")
    for g in (gc, gm, gr, gw):
        g.check(torch.ones(g.shape, dtype=torch.bool, device="cuda"), "calibration output")


@pytest.mark.parametrize("name", list(CASES))
def test_canary_score_select_compact(name):
    w, inp, gcache = _setup(name, seed=1, pos=(name == "bf16_d128"))
    S, n_cap, P, W, B = w.n_slices, w.n_cap, w.n_prompt, w.n_recent, w.budget
    c = tri.calibrate_centers(inp.q, w.group)
    gs = Guarded((S, n_cap), torch.float32)
    tri.score(gcache.kv, c, w.theta, w.offsets, inp.p_cur, gs.t, n_prompt=P, n_recent=W)
    j = torch.arange(n_cap, device="cuda")[None, :]
    nv = torch.as_tensor(gcache.nv0, device="cuda")[:, None]
    gs.check((j >= P) & (j < nv - W), "tri_score scores")
    gcache.check_untouched("tri_score")
    gs.snap()
    gk = Guarded((S, B), torch.int32)
    tri.select_topk(gs.t, gcache.kv, P, W, B, gk.t)
    gs.check(None, "tri_select_topk scores")
    gk.check(torch.ones(S, B, dtype=torch.bool, device="cuda"), "tri_select_topk keep")
    gcache.check_untouched("tri_select_topk")
    gk.snap()
    tri.compact_kv(gcache.kv, gk.t, B)
    gk.check(None, "tri_compact_kv keep")
    gcache.check_compacted(B, "tri_compact_kv")


@pytest.mark.parametrize("name", list(CASES))
def test_canary_compress_and_select_compact(name):
    w, inp, gcache = _setup(name, seed=2)
    S, n_cap, P, W, B = w.n_slices, w.n_cap, w.n_prompt, w.n_recent, w.budget
    c = tri.calibrate_centers(inp.q, w.group)
    need = tri.compress_workspace_bytes(gcache.kv)
    gw = Guarded((need,), torch.uint8)
    gk = Guarded((S, B), torch.int32)
    tri.compress(gcache.kv, c, w.theta, w.offsets, inp.p_cur, P, W, B, gk.t, workspace=gw.t)
    gw.check(torch.ones(need, dtype=torch.bool, device="cuda"), "tri_compress workspace")
    gk.check(torch.ones(S, B, dtype=torch.bool, device="cuda"), "tri_compress keep")
    gcache.check_compacted(B, "tri_compress")
    # tri_select_compact on a fresh cache, from scores that must stay as they are
    w, inp, gcache = _setup(name, seed=3)
    gs = Guarded((S, n_cap), torch.float32, torch.randn(S, n_cap))
    gk = Guarded((S, B), torch.int32)
    tri.select_compact(gs.t, gcache.kv, P, W, B, gk.t)
    gs.check(None, "tri_select_compact scores")
    gk.check(torch.ones(S, B, dtype=torch.bool, device="cuda"), "tri_select_compact keep")
    gcache.check_compacted(B, "tri_select_compact")


@pytest.mark.parametrize("name", list(CASES))
def test_canary_random_eviction(name):
    w, inp, gcache = _setup(name, seed=4)
    S, P, B = w.n_slices, w.n_prompt, w.budget
    for scope in (0, 1, 2):
        gk = Guarded((S, B), torch.int32)
        tri.rand_evict_scoped(gcache.kv, 5, scope, scope, P, 0, B, gk.t)
        gk.check(torch.ones(S, B, dtype=torch.bool, device="cuda"), "rand_evict_scoped keep")
        gcache.check_untouched("rand_evict_scoped")
    gk.snap()
    tri.compact_kv(gcache.kv, gk.t, B)
    gcache.check_compacted(B, "tri_compact_kv after rand_evict")
    w, inp, gcache = _setup(name, seed=5)
    gk = Guarded((S, B), torch.int32)
    tri.rand_evict_compact(gcache.kv, 9, 1, P, 0, B, gk.t)
    gk.check(torch.ones(S, B, dtype=torch.bool, device="cuda"), "rand_evict_compact keep")
    gcache.check_compacted(B, "rand_evict_compact")


@pytest.mark.parametrize("name", list(CASES))
def test_canary_gqa(name):
    w, inp, gcache = _setup(name, seed=6)
    S, n_cap, P, W, B, G = w.n_slices, w.n_cap, w.n_prompt, w.n_recent, w.budget, 3
    cq = tri.calibrate_centers(synth.make_inputs(synth.scaled(w, group=G), "cuda").q, 1)
    gsg = Guarded((S, G, n_cap), torch.float32)
    gst = Guarded((S, G, 2), torch.float32)
    need = tri.score_heads_workspace_bytes(gcache.kv, G)
    gw = Guarded((need,), torch.uint8)
    tri.score_heads(gcache.kv, cq, G, w.theta, w.offsets, inp.p_cur, gsg.t, gst.t, workspace=gw.t)
    j = torch.arange(n_cap, device="cuda")[None, None, :]
    nv = torch.as_tensor(gcache.nv0, device="cuda")[:, None, None]
    gsg.check((j < nv).expand(S, G, n_cap), "tri_score_heads scores")
    gst.check(torch.ones(S, G, 2, dtype=torch.bool, device="cuda"), "tri_score_heads stats")
    gw.check(torch.ones(need, dtype=torch.bool, device="cuda"), "tri_score_heads workspace")
    gcache.check_untouched("tri_score_heads")
    gsg.snap()
    gst.snap()
    gk = Guarded((S, B), torch.int32)
    gf = Guarded((S, n_cap), torch.float32)
    tri.select_topk_zmax(gsg.t, gst.t, G, gcache.kv, P, W, B, gk.t, final_scores=gf.t)
    gsg.check(None, "tri_select_topk_zmax scores")
    gst.check(None, "tri_select_topk_zmax stats")
    gk.check(torch.ones(S, B, dtype=torch.bool, device="cuda"), "tri_select_topk_zmax keep")
    gf.check((torch.arange(n_cap, device="cuda")[None, :] < torch.as_tensor(gcache.nv0, device="cuda")[:, None]),
             "tri_select_topk_zmax final scores")
    gcache.check_untouched("tri_select_topk_zmax")


@pytest.mark.parametrize("name", list(CASES))
def test_canary_union(name):
    w = CASES[name]
    inp = synth.make_inputs(w, "cuda")
    S, n_cap, P, W, B, H = w.n_slices, w.n_cap, w.n_prompt, w.n_recent, w.budget, w.n_kv_heads
    groups = S // H
    # every head of a (seq, layer) holds the same row count; the groups are ragged
    nv = _ragged(groups, n_cap, B, 8).repeat_interleave(H)
    gcache = GuardedCache(inp.k, inp.v, nv)
    c = tri.calibrate_centers(inp.q, w.group)
    gs = Guarded((S, n_cap), torch.float32, torch.zeros(S, n_cap))
    tri.score(gcache.kv, c, w.theta, w.offsets, inp.p_cur, gs.t)
    gs.snap()
    k_head = (B - P - W) // 2
    need = tri.select_union_workspace_bytes(gcache.kv, P, W, k_head)
    gw = Guarded((need,), torch.uint8)
    gk = Guarded((S, B), torch.int32)
    gf = Guarded((groups, n_cap), torch.float32)
    tri.select_union(gs.t, gcache.kv, P, W, B, k_head, gk.t, final_scores=gf.t, workspace=gw.t)
    gs.check(None, "tri_select_union scores")
    gw.check(torch.ones(need, dtype=torch.bool, device="cuda"), "tri_select_union workspace")
    gk.check(torch.ones(S, B, dtype=torch.bool, device="cuda"), "tri_select_union keep")
    nvg = torch.as_tensor(nv[::H].numpy(), device="cuda")[:, None]
    gf.check(torch.arange(n_cap, device="cuda")[None, :] < nvg, "tri_select_union final scores")
    gcache.check_untouched("tri_select_union")


def test_canary_paged_blocks_used():
    w = CASES["bf16_d128"]
    inp = synth.make_inputs(w, "cuda")
    bs = 16
    n_seq, L, H, n_cap, d = inp.k.shape
    mb = -(-n_cap // bs)
    kp = torch.zeros(n_seq * mb, L, H, bs, d, dtype=inp.k.dtype, device="cuda")
    table = torch.arange(n_seq * mb, dtype=torch.int32, device="cuda").view(n_seq, mb)
    nv = _ragged(w.n_slices, mb * bs, w.budget, 9).to("cuda")
    kv = tri.PagedKVCache(kp, kp.clone(), table, nv, None, None)
    go = Guarded((n_seq,), torch.int32)
    tri.paged_blocks_used(kv, go.t)
    go.check(torch.ones(n_seq, dtype=torch.bool, device="cuda"), "tri_paged_blocks_used")
    most = nv.view(n_seq, -1).max(dim=1).values
    assert torch.equal(go.t, (most + bs - 1) // bs)
