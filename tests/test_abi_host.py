"""Host-only checks of the C ABI: the library builds and loads, exports every
function include/tri.h declares, and rejects bad arguments on the host (these
calls return before anything touches CUDA, so no GPU is needed)."""
import ctypes
import os
import re

import pytest

from kv_cache_compression_tri_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    import kv_cache_compression_tri_gb300 as tri
    return tri.load_library()


def _declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        txt = open(os.path.join(ROOT, "include", h)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        txt = re.sub(r"//[^\n]*", "", txt)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", txt, flags=re.M):
            if m.group(1) not in ("if", "while", "for", "return", "sizeof"):
                names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("tri_calibrate_centers", "tri_score", "tri_select_topk", "tri_compact_kv",
              "rand_evict", "tri_status_string", "tri_launch_count"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = os.popen(f"nm -D --defined-only {_build.LIB}").read()
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in _declared_functions() if n not in exported]
    assert not missing, missing
    for n in _declared_functions():
        getattr(lib, n)


def test_status_strings_and_version(lib):
    for code in range(5):
        assert lib.tri_status_string(code)
    assert lib.tri_status_string(99) == b"unknown status"
    assert lib.tri_abi_version() == 3
    assert lib.tri_launch_count() >= 0


def _kv(**over):
    import kv_cache_compression_tri_gb300 as tri
    f = dict(k=0x10000, v=0x20000, pos=None, pos_out=0x30000, n_valid=0x40000, slice_stride=128 * 64,
             n_seq=1, n_layers=1, n_kv_heads=2, n_cap=128, head_dim=64, dtype=1, dev_status=None,
             key_layout=0, block_table=None, block_size=0, num_blocks=0, block_stride=0, layer_stride=0,
             head_stride=0)
    f.update(over)
    return tri._TriKV(f["k"], f["v"], f["pos"], f["pos_out"], f["n_valid"], f["slice_stride"],
                      f["n_seq"], f["n_layers"], f["n_kv_heads"], f["n_cap"], f["head_dim"], f["dtype"],
                      f["dev_status"], f["key_layout"], f["block_table"], f["block_size"], f["num_blocks"],
                      f["block_stride"], f["layer_stride"], f["head_stride"])


PAGED = dict(block_table=0xF0000, block_size=16, num_blocks=64, block_stride=2 * 16 * 64, layer_stride=2 * 16 * 64,
             head_stride=16 * 64, slice_stride=0)


INVALID, UNSUPPORTED = 1, 2


@pytest.mark.parametrize("over,code", [
    (dict(head_dim=96), UNSUPPORTED),
    (dict(dtype=7), UNSUPPORTED),
    (dict(k=None), INVALID),
    (dict(k=0x10008), INVALID),  # not 16-byte aligned
    (dict(n_valid=None), INVALID),
    (dict(slice_stride=100), INVALID),  # < n_cap * head_dim
    (dict(slice_stride=128 * 64 + 4), INVALID),  # rows not 16-byte aligned
    (dict(n_cap=0), INVALID),
    (dict(n_seq=0), INVALID),
    (dict(pos_out=None), INVALID),  # compaction needs a position target
    (dict(key_layout=2), INVALID),  # neither pre- nor post-RoPE
    (dict(PAGED, block_size=24), INVALID),  # not a power of two
    (dict(PAGED, block_size=48), INVALID),
    (dict(PAGED, block_size=8), INVALID),  # below 16 rows
    (dict(PAGED, block_size=256), INVALID),  # n_cap 128 not a whole number of blocks
    (dict(PAGED, num_blocks=0), INVALID),
    (dict(PAGED, head_stride=4), INVALID),  # rows of one head overlap the next head's
    (dict(PAGED, block_stride=2 * 16 * 64 + 2), INVALID),  # blocks not 16-byte aligned
    (dict(PAGED, block_table=0xF0002), INVALID),
])
def test_compact_rejects_bad_cache(lib, over, code):
    kv = _kv(**over)
    assert lib.tri_compact_kv(ctypes.byref(kv), 0x50000, 64, None) == code


def test_select_rejects_bad_budget(lib):
    kv = _kv()
    assert lib.tri_select_topk(0x60000, ctypes.byref(kv), 40, 40, 64, 0x50000, None) == INVALID
    assert lib.tri_select_topk(0x60000, ctypes.byref(kv), -1, 0, 64, 0x50000, None) == INVALID
    assert lib.tri_select_topk(0x60000, ctypes.byref(kv), 0, 0, 0, 0x50000, None) == INVALID
    assert lib.tri_select_topk(0x60000, ctypes.byref(kv), 0, 0, 129, 0x50000, None) == INVALID
    assert lib.tri_select_topk(None, ctypes.byref(kv), 0, 0, 64, 0x50000, None) == INVALID
    assert lib.tri_select_topk(0x60000, None, 0, 0, 64, 0x50000, None) == INVALID
    assert lib.rand_evict(ctypes.byref(kv), 0, 0, 40, 40, 64, 0x50000, None) == INVALID
    assert lib.rand_evict(ctypes.byref(_kv(n_layers=70000)), 0, 0, 0, 0, 64, 0x50000, None) == INVALID
    assert lib.rand_evict_scoped(ctypes.byref(kv), 0, 0, 3, 0, 0, 64, 0x50000, None) == INVALID  # no such scope


def test_score_rejects_bad_args(lib):
    import kv_cache_compression_tri_gb300 as tri
    kv = _kv()
    c = tri._TriCenters(0x70000, 0x80000, 0x90000)
    offs = (ctypes.c_int32 * 3)(1, 2, 4)
    op = ctypes.cast(offs, ctypes.c_void_p)
    call = lambda **o: lib.tri_score(ctypes.byref(o.get("kv", kv)), ctypes.byref(o.get("c", c)),
                                     o.get("theta", 1e4), o.get("style", 0), o.get("norm", 0),
                                     o.get("offs", op), o.get("n_off", 3), o.get("p_cur", 0xA0000),
                                     0, 0, o.get("scores", 0xB0000), None)
    assert call(theta=0.5) == INVALID
    assert call(theta=float("nan")) == INVALID
    assert call(n_off=0) == INVALID
    assert call(n_off=65) == INVALID
    assert call(offs=None) == INVALID
    assert call(style=5) == INVALID
    assert call(norm=3) == INVALID
    assert call(p_cur=None) == INVALID
    assert call(scores=None) == INVALID
    assert call(kv=_kv(head_dim=256)) == UNSUPPORTED
    assert call(kv=_kv(key_layout=-1)) == INVALID
    assert call(c=tri._TriCenters(None, 0x80000, 0x90000)) == INVALID


def test_calibrate_rejects_bad_args(lib):
    import kv_cache_compression_tri_gb300 as tri
    c = tri._TriCenters(0x70000, 0x80000, 0x90000)
    ws = lib.tri_calibrate_workspace_bytes(2, 8, 4, 128, 4096)
    assert ws > 0
    assert lib.tri_calibrate_workspace_bytes(2, 8, 3, 128, 4096) == 0  # 8 % 3 != 0
    f = lib.tri_calibrate_centers
    assert f(0x10000, 1, 2, 8, 3, 128, 4096, 0, c, 0xC0000, ws, None) == INVALID
    assert f(0x10000, 1, 2, 8, 4, 96, 4096, 0, c, 0xC0000, ws, None) == UNSUPPORTED
    assert f(0x10000, 1, 2, 8, 4, 128, 4096, 0, c, 0xC0000, ws - 1, None) == INVALID
    assert f(0x10000, 1, 2, 8, 4, 128, 4096, 0, c, None, ws, None) == INVALID
    assert f(0x10004, 1, 2, 8, 4, 128, 4096, 0, c, 0xC0000, ws, None) == INVALID


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import kv_cache_compression_tri_gb300 as tri
    monkeypatch.setattr(tri, "_lib", None)
    monkeypatch.setattr(tri, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        tri.load_library()


def test_kv_cache_bytes_worked_example(golden):
    from kv_cache_compression_tri_gb300.synth import kv_cache_bytes
    for c in golden("kv_bytes.json")["cases"]:
        assert kv_cache_bytes(c["layers"], c["d_model"], c["tokens"], c["elem_bytes"], c["batch"]) == c["bytes"]


def test_gqa_entry_points_reject_bad_args(lib):
    import kv_cache_compression_tri_gb300 as tri
    kv = _kv()
    c = tri._TriCenters(0x70000, 0x80000, 0x90000)
    offs = (ctypes.c_int32 * 3)(1, 2, 4)
    op = ctypes.cast(offs, ctypes.c_void_p)
    ws = lib.tri_score_heads_workspace_bytes(ctypes.byref(kv), 4)
    assert ws > 0 and ws % 8 == 0
    assert lib.tri_score_heads_workspace_bytes(ctypes.byref(kv), 9) == 0  # group > 8
    assert lib.tri_score_heads_workspace_bytes(ctypes.byref(kv), 0) == 0
    call = lambda **o: lib.tri_score_heads(ctypes.byref(kv), ctypes.byref(c), o.get("group", 4), 1e4, 0, 0, op,
                                           3, 0xA0000, 0xB0000, o.get("stats", 0xD0000),
                                           o.get("ws", 0xC0000), o.get("ws_bytes", ws), None)
    assert call(group=9) == INVALID
    assert call(stats=None) == INVALID
    assert call(ws=None) == INVALID
    assert call(ws_bytes=ws - 1) == INVALID
    sel = lambda **o: lib.tri_select_topk_zmax(0xB0000, o.get("stats", 0xD0000), o.get("group", 4),
                                               ctypes.byref(kv), 0, 0, o.get("budget", 64), 0x50000,
                                               o.get("final", None), None)
    assert sel(group=0) == INVALID
    assert sel(stats=None) == INVALID
    assert sel(budget=129) == INVALID
    assert sel(final=0xE0002) == INVALID  # misaligned output


def test_paged_blocks_used_needs_a_paged_cache(lib):
    assert lib.tri_paged_blocks_used(ctypes.byref(_kv()), 0x50000, None) == INVALID
    assert lib.tri_paged_blocks_used(ctypes.byref(_kv(**PAGED)), None, None) == INVALID


def test_wait_timeout_selftest_rejects_bad_args(lib):
    f = lib.tri_selftest_wait_timeout
    assert f(None, 1000000, None) == INVALID  # no status word
    assert f(0x10002, 1000000, None) == INVALID  # misaligned status word
    assert f(0x10000, 999, None) == INVALID  # limit below 1 us
    assert f(0x10000, 1000000001, None) == INVALID  # limit above 1 s


def test_compress_rejects_bad_args(lib):
    import kv_cache_compression_tri_gb300 as tri
    kv = _kv()
    c = tri._TriCenters(0x70000, 0x80000, 0x90000)
    offs = (ctypes.c_int32 * 3)(1, 2, 4)
    op = ctypes.cast(offs, ctypes.c_void_p)
    cws = lib.tri_compress_workspace_bytes(ctypes.byref(kv))
    assert cws == 2 * 128 * 4  # the scores
    comp = lambda **o: lib.tri_compress(ctypes.byref(o.get("kv", kv)), ctypes.byref(c), 1e4, 0, 0, op, 3, 0xA0000,
                                        o.get("P", 0), o.get("W", 0), o.get("budget", 64), o.get("keep", 0x50000),
                                        o.get("ws", 0xC0000), o.get("ws_bytes", cws), None)
    assert comp(ws_bytes=cws - 1) == INVALID
    assert comp(ws=None) == INVALID
    assert comp(ws=0xC0008) == INVALID  # the scores need 16-byte alignment
    assert comp(keep=None) == INVALID
    assert comp(P=40, W=40) == INVALID  # protected rows above the budget
    assert comp(budget=129) == INVALID  # budget above n_cap
    assert comp(kv=_kv(pos_out=None)) == INVALID
    assert comp(kv=_kv(dtype=7)) == UNSUPPORTED
    assert comp(kv=_kv(head_dim=96)) == UNSUPPORTED
