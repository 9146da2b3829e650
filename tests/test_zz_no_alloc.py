"""tri_calibrate_centers_noalloc: calibration for callers that cannot allocate
device memory (for example a plugin inside an engine that owns all device
memory through its own pool, or latency-critical code that must not call
cudaMalloc/cudaFree because they can synchronise the device). It keeps its
partial sums in a fixed array inside the library instead of caller scratch.

The test calls it through the C ABI twice in a row on different inputs and
compares each result with tri_calibrate_centers (the entry point that takes
caller scratch), within the calibration tolerance the other tests use. It
also checks that an oversized shape is refused. This file is named so that
pytest collects it last."""
import ctypes

import pytest
import torch

import kv_cache_compression_tri_gb300 as tri
from kv_cache_compression_tri_gb300 import synth

pytestmark = pytest.mark.gpu

CALIB_TOL = 1e-5
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


def _close(a: tri.Centers, b: tri.Centers):
    m = b.mean_norm
    assert torch.all(torch.abs(a.center - b.center) <= CALIB_TOL * m[..., None])
    assert torch.all(torch.abs(a.mean_norm - m) <= CALIB_TOL * m)
    assert torch.all(torch.abs(a.mrl - b.mrl) <= CALIB_TOL)


def test_noalloc_matches_scratch_entry_point_twice(lib):
    cases = [
        (synth.scaled(synth.WORKLOADS["qwen3_8b_stack"], n_layers=6, n_cal=2048), 0),
        (synth.WORKLOADS["qwen3_8b_layer"], 1),
    ]
    for w, style in cases:  # two calls in a row: the second must not see the first's partials
        inp = synth.make_inputs(w, "cuda", seqs=1)
        ref = tri.calibrate_centers(inp.q, w.group, style=style)
        got = _noalloc(lib, inp.q, w.group, style)
        torch.cuda.synchronize()
        _close(got, ref)


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    # 128 layers x 64 KV heads x 64 bands x 3 partial sums x 4 B = 6.3 MB > 4 MiB
    need = lib.tri_calibrate_workspace_bytes(128, 64, 1, 128, 4096)
    assert need > MAX_SCRATCH
    q = torch.zeros(16, dtype=torch.uint8, device="cuda")
    out = _outputs(1, 1, 64)
    st = lib.tri_calibrate_centers_noalloc(q.data_ptr(), 1, 128, 64, 1, 128, 4096, 0, out._abi(),
                                           torch.cuda.current_stream().cuda_stream)
    assert st == INVALID_ARG
