"""The failure path the kernels share, on the GPU without a fault: a bounded
mbarrier wait that nothing completes runs out, records TRI_DEV_TIMEOUT in the
caller's status word (first error wins) and returns; the context stays
usable and the next calls run normally."""
import time

import numpy as np
import pytest
import torch

import kv_cache_compression_tri_gb300 as tri
from kv_cache_compression_tri_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    tri.load_library()


def test_bounded_wait_runs_out_and_reports_timeout():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    tri.selftest_wait_timeout(status, 20_000_000)  # 20 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == tri.DEV_TIMEOUT
    assert elapsed >= 0.018  # the wait lasted its limit
    # first error wins: an earlier code is kept
    status.fill_(tri.DEV_NAN_SCORE)
    tri.selftest_wait_timeout(status, 1000)
    torch.cuda.synchronize()
    assert int(status.item()) == tri.DEV_NAN_SCORE


def test_context_usable_after_a_timeout():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tri.selftest_wait_timeout(status, 5_000_000)
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w, "cuda")
    c = tri.calibrate_centers(inp.q, w.group)
    kv = tri.KVCache(inp.k, inp.v, inp.n_valid.clone(), None,
                     torch.full((w.n_slices, w.n_cap), -1, dtype=torch.int32, device="cuda"),
                     torch.zeros(1, dtype=torch.int32, device="cuda"))
    scores = torch.full((w.n_slices, w.n_cap), float("nan"), device="cuda")
    tri.score(kv, c, w.theta, w.offsets, inp.p_cur, scores, n_prompt=0, n_recent=0)
    keep = torch.empty(w.n_slices, w.budget, dtype=torch.int32, device="cuda")
    tri.select_topk(scores, kv, w.n_prompt, w.n_recent, w.budget, keep)
    torch.cuda.synchronize()
    assert int(status.item()) == tri.DEV_TIMEOUT
    assert int(kv.dev_status.item()) == 0
    n = int(inp.n_valid[0].item())
    assert torch.isfinite(scores[:, :n]).all()
    k0 = keep[0].cpu().numpy()
    assert np.all(np.diff(k0[k0 >= 0]) > 0)
