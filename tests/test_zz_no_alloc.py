"""tri_calibrate_centers_noalloc: calibration for callers that cannot allocate
device memory (for example a plugin inside an engine that owns all device
memory through its own pool, or latency-critical code that must not call
cudaMalloc/cudaFree because they can synchronise the device). It keeps its
partial sums in a fixed array inside the library instead of caller scratch.

The test calls it through the C ABI twice in a row on different inputs and
compares each result with tri_calibrate_centers (the entry point that takes
caller scratch). Both run the same kernels with the same split count, so the
results must be bit-identical. It covers bf16 and fp32 queries, the largest
shape whose scratch still fits the library's array, and the refusal of the
next larger one. This file is named so that pytest collects it last."""
import ctypes

import pytest
import torch

import kv_cache_compression_tri_gb300 as tri
from kv_cache_compression_tri_gb300 import synth

pytestmark = pytest.mark.gpu

INVALID_ARG = 1
MAX_SCRATCH = 4 * 1024 * 1024


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    lib = tri.load_library()
    f = lib.tri_calibrate_centers_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_int64, ctypes.c_int, tri._TriCenters, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


def _outputs(L, H, F):
    return tri.Centers(torch.full((L * H, F, 2), float("nan"), device="cuda"),
                       torch.full((L * H, F), float("nan"), device="cuda"),
                       torch.full((L * H, F), float("nan"), device="cuda"))


def _noalloc(lib, q, group, style):
    L, Hq, n_tok, d = q.shape
    out = _outputs(L, Hq // group, d // 2)
    dt = 1 if q.dtype == torch.bfloat16 else 0
    st = lib.tri_calibrate_centers_noalloc(q.data_ptr(), dt, L, Hq, group, d, n_tok, style, out._abi(),
                                           torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.tri_status_string(st)
    return out


def _same(a: tri.Centers, b: tri.Centers):
    # Same kernels, same split count, same order of additions: same bits.
    assert torch.equal(a.center, b.center)
    assert torch.equal(a.mean_norm, b.mean_norm)
    assert torch.equal(a.mrl, b.mrl)


def test_noalloc_matches_scratch_entry_point_twice(lib):
    cases = [
        (synth.scaled(synth.WORKLOADS["qwen3_8b_stack"], n_layers=6, n_cal=2048), 0),
        (synth.WORKLOADS["qwen3_8b_layer"], 1),
        (synth.WORKLOADS["tiny"], 0),  # fp32 queries
    ]
    for w, style in cases:  # calls in a row: none may see an earlier call's partials
        inp = synth.make_inputs(w, "cuda", seqs=1)
        ref = tri.calibrate_centers(inp.q, w.group, style=style)
        got = _noalloc(lib, inp.q, w.group, style)
        torch.cuda.synchronize()
        _same(got, ref)


def test_noalloc_accepts_the_largest_shape_that_fits(lib):
    # 43 layers x 127 KV heads x 64 bands x 3 sums x 4 B (one split each) =
    # 4,194,048 B, just under the 4 MiB array; one more head does not fit.
    L, H, d, n_tok = 43, 127, 128, 16
    need = lib.tri_calibrate_workspace_bytes(L, H, 1, d, n_tok)
    assert need <= MAX_SCRATCH and need + 64 * 3 * 4 > MAX_SCRATCH
    g = torch.Generator(device="cpu").manual_seed(5)
    q = (torch.randn(L, H, n_tok, d, generator=g) * 2.0 + 0.5).to(torch.bfloat16).cuda()
    ref = tri.calibrate_centers(q, 1, style=0)
    got = _noalloc(lib, q, 1, 0)
    torch.cuda.synchronize()
    _same(got, ref)
    assert lib.tri_calibrate_workspace_bytes(1, L * H + 1, 1, d, n_tok) > MAX_SCRATCH
    out = _outputs(1, L * H + 1, d // 2)
    q1 = torch.zeros(1, L * H + 1, n_tok, d, dtype=torch.bfloat16, device="cuda")
    st = lib.tri_calibrate_centers_noalloc(q1.data_ptr(), 1, 1, L * H + 1, 1, d, n_tok, 0, out._abi(),
                                           torch.cuda.current_stream().cuda_stream)
    assert st == INVALID_ARG


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    # 128 layers x 64 KV heads x 64 bands x 3 partial sums x 4 B = 6.3 MB > 4 MiB
    need = lib.tri_calibrate_workspace_bytes(128, 64, 1, 128, 4096)
    assert need > MAX_SCRATCH
    q = torch.zeros(16, dtype=torch.uint8, device="cuda")
    out = _outputs(1, 1, 64)
    st = lib.tri_calibrate_centers_noalloc(q.data_ptr(), 1, 128, 64, 1, 128, 4096, 0, out._abi(),
                                           torch.cuda.current_stream().cuda_stream)
    assert st == INVALID_ARG
