"""GB300 KV-cache compression: TriAttention scoring, budgeted selection,
in-place compaction, and Random Attention eviction.

This module is a thin ctypes binding over ``libtri.so`` (C ABI in
``include/tri.h``): it turns torch tensors into device pointers and the
current CUDA stream into a stream handle, and raises on a non-zero status.
Every step of the path runs in the library's CUDA kernels; there is no
fallback. If the library has not been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

from ._build import LIB as _LIB_PATH

__all__ = [
    "TriError", "KVCache", "PagedKVCache", "select_compact", "rand_evict_compact", "paged_blocks_used", "Centers", "lib_path", "load_library", "calibrate_centers",
    "calibrate_workspace_bytes", "score", "select_topk", "compact_kv", "rand_evict",
    "compress", "compress_workspace_bytes", "score_heads", "score_heads_workspace_bytes",
    "select_topk_zmax", "select_union", "select_union_workspace_bytes", "rand_evict_scoped", "DRAW_PER_HEAD", "DRAW_PER_LAYER", "DRAW_PER_SEQUENCE",
    "launch_count", "ROPE_INTERLEAVED", "ROPE_HALF", "NORM_WEIGHTED", "NORM_UNWEIGHTED",
    "DEV_OK", "DEV_NVALID_OVER_CAP", "DEV_NAN_SCORE", "DEV_BAD_KEEP",
]

ROPE_INTERLEAVED, ROPE_HALF = 0, 1
NORM_WEIGHTED, NORM_UNWEIGHTED = 0, 1
F32, BF16 = 0, 1
DEV_OK, DEV_NVALID_OVER_CAP, DEV_NAN_SCORE, DEV_BAD_KEEP, DEV_TIMEOUT, DEV_GROUP_NVALID, DEV_BAD_BLOCK = (
    0, 1, 2, 3, 4, 5, 6)

_DTYPES = {torch.float32: F32, torch.bfloat16: BF16}


class TriError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


class _TriKV(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("pos", ctypes.c_void_p),
        ("pos_out", ctypes.c_void_p), ("n_valid", ctypes.c_void_p),
        ("slice_stride", ctypes.c_int64), ("n_seq", ctypes.c_int32),
        ("n_layers", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("n_cap", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int),
        ("dev_status", ctypes.c_void_p), ("key_layout", ctypes.c_int),
        ("block_table", ctypes.c_void_p), ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
        ("block_stride", ctypes.c_int64), ("layer_stride", ctypes.c_int64), ("head_stride", ctypes.c_int64),
    ]


class _TriCenters(ctypes.Structure):
    _fields_ = [("center", ctypes.c_void_p), ("mean_norm", ctypes.c_void_p),
                ("mrl", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libtri.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libtri.so is not built ({_LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i32, i64, u32, u64 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_uint32, ctypes.c_uint64)
        kvp = ctypes.POINTER(_TriKV)
        lib.tri_status_string.argtypes = [ctypes.c_int]
        lib.tri_status_string.restype = ctypes.c_char_p
        lib.tri_abi_version.restype = i32
        lib.tri_launch_count.restype = u64
        lib.tri_calibrate_workspace_bytes.argtypes = [i32, i32, i32, i32, i64]
        lib.tri_calibrate_workspace_bytes.restype = ctypes.c_size_t
        lib.tri_calibrate_centers.argtypes = [vp, ctypes.c_int, i32, i32, i32, i32, i64,
                                              ctypes.c_int, _TriCenters, vp, ctypes.c_size_t, vp]
        lib.tri_calibrate_centers.restype = ctypes.c_int
        lib.tri_score.argtypes = [kvp, ctypes.POINTER(_TriCenters), ctypes.c_double, ctypes.c_int,
                                  ctypes.c_int, vp, i32, vp, i32, i32, vp, vp]
        lib.tri_score.restype = ctypes.c_int
        lib.tri_select_topk.argtypes = [vp, kvp, i32, i32, i32, vp, vp]
        lib.tri_select_topk.restype = ctypes.c_int
        lib.tri_compact_kv.argtypes = [kvp, vp, i32, vp]
        lib.tri_compact_kv.restype = ctypes.c_int
        lib.rand_evict.argtypes = [kvp, u64, u32, i32, i32, i32, vp, vp]
        lib.rand_evict.restype = ctypes.c_int
        lib.rand_evict_scoped.argtypes = [kvp, u64, u32, ctypes.c_int, i32, i32, i32, vp, vp]
        lib.rand_evict_scoped.restype = ctypes.c_int
        lib.tri_compress_workspace_bytes.argtypes = [kvp]
        lib.tri_compress_workspace_bytes.restype = ctypes.c_size_t
        lib.tri_compress.argtypes = [kvp, ctypes.POINTER(_TriCenters), ctypes.c_double, ctypes.c_int,
                                     ctypes.c_int, vp, i32, vp, i32, i32, i32, vp, vp, ctypes.c_size_t, vp]
        lib.tri_compress.restype = ctypes.c_int
        lib.tri_score_heads_workspace_bytes.argtypes = [kvp, i32]
        lib.tri_score_heads_workspace_bytes.restype = ctypes.c_size_t
        lib.tri_score_heads.argtypes = [kvp, ctypes.POINTER(_TriCenters), i32, ctypes.c_double, ctypes.c_int,
                                        ctypes.c_int, vp, i32, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.tri_score_heads.restype = ctypes.c_int
        lib.tri_select_topk_zmax.argtypes = [vp, vp, i32, kvp, i32, i32, i32, vp, vp, vp]
        lib.tri_select_topk_zmax.restype = ctypes.c_int
        lib.tri_select_union_workspace_bytes.argtypes = [kvp, i32, i32, i32]
        lib.tri_select_union_workspace_bytes.restype = ctypes.c_size_t
        lib.tri_select_union.argtypes = [vp, kvp, i32, i32, i32, i32, vp, vp, vp, ctypes.c_size_t, vp]
        lib.tri_select_union.restype = ctypes.c_int
        lib.tri_select_compact.argtypes = [vp, kvp, i32, i32, i32, vp, vp]
        lib.tri_select_compact.restype = ctypes.c_int
        lib.rand_evict_compact.argtypes = [kvp, u64, u32, ctypes.c_int, i32, i32, i32, vp, vp]
        lib.rand_evict_compact.restype = ctypes.c_int
        lib.tri_paged_blocks_used.argtypes = [kvp, vp, vp]
        lib.tri_paged_blocks_used.restype = ctypes.c_int
        lib.tri_selftest_wait_timeout.argtypes = [vp, u64, vp]
        lib.tri_selftest_wait_timeout.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != 0:
        msg = load_library().tri_status_string(status).decode()
        raise TriError(fn, status, msg)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def launch_count() -> int:
    """Kernels the library has launched in this process."""
    return int(load_library().tri_launch_count())


@dataclass
class Centers:
    """Per-(layer, KV head) query statistics (fp32, device): center
    [L*H][F][2], mean_norm [L*H][F], mrl [L*H][F]."""
    center: torch.Tensor
    mean_norm: torch.Tensor
    mrl: torch.Tensor

    def _abi(self) -> _TriCenters:
        for t in (self.center, self.mean_norm, self.mrl):
            assert t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()
        return _TriCenters(self.center.data_ptr(), self.mean_norm.data_ptr(), self.mrl.data_ptr())


@dataclass
class KVCache:
    """A batch of caches: k, v [n_seq, n_layers, n_kv_heads, n_cap, head_dim]
    (bf16 or fp32, device); n_valid [S] int32; pos / pos_out [S, n_cap] int32
    (pos may be None: position = slot index); dev_status [1] int32.
    post_rope: k holds RoPE-rotated keys (the score then ignores pos)."""
    k: torch.Tensor
    v: torch.Tensor
    n_valid: torch.Tensor
    pos: torch.Tensor | None
    pos_out: torch.Tensor | None
    dev_status: torch.Tensor | None = None
    post_rope: bool = False

    @property
    def shape(self):
        return tuple(self.k.shape)

    @property
    def n_slices(self) -> int:
        s = self.k.shape
        return s[0] * s[1] * s[2]

    @property
    def n_cap(self) -> int:
        return self.k.shape[3]

    @property
    def device(self):
        return self.k.device

    def _abi(self) -> _TriKV:
        n_seq, L, H, n_cap, d = self.k.shape
        assert self.k.is_cuda and self.k.dtype in _DTYPES
        assert self.v.shape == self.k.shape and self.v.dtype == self.k.dtype
        # rows contiguous, slices evenly strided
        assert self.k.stride(4) == 1 and self.k.stride(3) == d
        stride = self.k.stride(2)
        assert self.k.stride(1) == H * stride and self.k.stride(0) == L * H * stride
        assert tuple(self.v.stride()) == tuple(self.k.stride())
        assert self.n_valid.dtype == torch.int32 and self.n_valid.numel() == n_seq * L * H
        for t in (self.pos, self.pos_out):
            if t is not None:
                assert t.dtype == torch.int32 and t.is_contiguous() and t.numel() == n_seq * L * H * n_cap
        return _TriKV(self.k.data_ptr(), self.v.data_ptr(), _ptr(self.pos), _ptr(self.pos_out),
                      self.n_valid.data_ptr(), stride, n_seq, L, H, n_cap, d, _DTYPES[self.k.dtype],
                      _ptr(self.dev_status), 1 if self.post_rope else 0, None, 0, 0, 0, 0, 0)


@dataclass
class PagedKVCache:
    """A paged batch of caches: k, v pools [num_blocks, n_layers, n_kv_heads,
    block_size, head_dim] (bf16 or fp32, device; any strides that keep each
    (block, layer, head) run of block_size rows contiguous); block_table
    [n_seq, blocks per sequence] int32 (physical block of each logical block,
    shared by the sequence's layers and heads); n_valid [S] int32; pos /
    pos_out [S, n_cap] int32 with n_cap = blocks per sequence * block_size."""
    k: torch.Tensor
    v: torch.Tensor
    block_table: torch.Tensor
    n_valid: torch.Tensor
    pos: torch.Tensor | None
    pos_out: torch.Tensor | None
    dev_status: torch.Tensor | None = None
    post_rope: bool = False

    @property
    def n_seq(self) -> int:
        return self.block_table.shape[0]

    @property
    def n_slices(self) -> int:
        return self.n_seq * self.k.shape[1] * self.k.shape[2]

    @property
    def n_cap(self) -> int:
        return self.block_table.shape[1] * self.k.shape[3]

    @property
    def device(self):
        return self.k.device

    def _abi(self) -> _TriKV:
        nb, L, H, bs, d = self.k.shape
        assert self.k.is_cuda and self.k.dtype in _DTYPES
        assert self.v.shape == self.k.shape and self.v.dtype == self.k.dtype
        assert tuple(self.v.stride()) == tuple(self.k.stride())
        assert self.k.stride(4) == 1 and self.k.stride(3) == d
        assert self.block_table.dtype == torch.int32 and self.block_table.is_contiguous()
        S, n_cap = self.n_slices, self.n_cap
        assert self.n_valid.dtype == torch.int32 and self.n_valid.numel() == S
        for t in (self.pos, self.pos_out):
            if t is not None:
                assert t.dtype == torch.int32 and t.is_contiguous() and t.numel() == S * n_cap
        return _TriKV(self.k.data_ptr(), self.v.data_ptr(), _ptr(self.pos), _ptr(self.pos_out),
                      self.n_valid.data_ptr(), 0, self.n_seq, L, H, n_cap, d, _DTYPES[self.k.dtype],
                      _ptr(self.dev_status), 1 if self.post_rope else 0, self.block_table.data_ptr(), bs, nb,
                      self.k.stride(0), self.k.stride(1), self.k.stride(2))


def paged_blocks_used(kv: PagedKVCache, out: torch.Tensor, stream=None) -> torch.Tensor:
    """Blocks each sequence still uses after compaction (tri_paged_blocks_used);
    table entries from there on are free. out: [n_seq] int32."""
    lib = load_library()
    assert out.dtype == torch.int32 and out.is_contiguous() and out.numel() == kv.n_seq
    kvs = kv._abi()
    _check("tri_paged_blocks_used", lib.tri_paged_blocks_used(ctypes.byref(kvs), out.data_ptr(), _stream(stream)))
    return out


def selftest_wait_timeout(status: torch.Tensor, limit_ns: int, stream=None) -> torch.Tensor:
    """The kernels' failure path (tri_selftest_wait_timeout): a bounded wait
    on an mbarrier nothing arrives on runs out after limit_ns and sets
    status (device int32 [1]) to DEV_TIMEOUT."""
    lib = load_library()
    assert status.dtype == torch.int32 and status.is_cuda and status.numel() >= 1
    _check("tri_selftest_wait_timeout", lib.tri_selftest_wait_timeout(status.data_ptr(), int(limit_ns),
                                                                      _stream(stream)))
    return status


def calibrate_workspace_bytes(n_layers: int, n_q_heads: int, group: int, head_dim: int,
                              n_tok: int) -> int:
    return int(load_library().tri_calibrate_workspace_bytes(n_layers, n_q_heads, group, head_dim, n_tok))


def calibrate_centers(q: torch.Tensor, group: int, style: int = ROPE_INTERLEAVED,
                      out: Centers | None = None, workspace: torch.Tensor | None = None,
                      stream=None) -> Centers:
    """Per-KV-head query centre, mean norm and MRL from pre-RoPE queries q
    [L, Hq, n_tok, d] (tri_calibrate_centers)."""
    lib = load_library()
    L, Hq, n_tok, d = q.shape
    assert q.is_cuda and q.is_contiguous() and q.dtype in _DTYPES
    H, F = Hq // group, d // 2
    if out is None:
        out = Centers(torch.empty(L * H, F, 2, device=q.device), torch.empty(L * H, F, device=q.device),
                      torch.empty(L * H, F, device=q.device))
    ws_bytes = calibrate_workspace_bytes(L, Hq, group, d, n_tok)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    assert workspace.numel() >= ws_bytes
    _check("tri_calibrate_centers", lib.tri_calibrate_centers(
        q.data_ptr(), _DTYPES[q.dtype], L, Hq, group, d, n_tok, style, out._abi(),
        workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return out


def score(kv: KVCache, centers: Centers, rope_theta: float, offsets, p_cur: torch.Tensor,
          scores: torch.Tensor, n_prompt: int = 0, n_recent: int = 0,
          style: int = ROPE_INTERLEAVED, norm_mode: int = NORM_WEIGHTED, stream=None) -> torch.Tensor:
    """Offset-averaged TriAttention score of rows [n_prompt, n_valid - n_recent)
    of every slice into scores [S, n_cap] fp32 (tri_score)."""
    lib = load_library()
    offs = (ctypes.c_int32 * len(offsets))(*[int(o) for o in offsets])
    assert p_cur.dtype == torch.int64 and p_cur.is_cuda
    assert scores.dtype == torch.float32 and scores.is_contiguous()
    assert scores.numel() == kv.n_slices * kv.n_cap
    kvs, cs = kv._abi(), centers._abi()
    _check("tri_score", lib.tri_score(ctypes.byref(kvs), ctypes.byref(cs), float(rope_theta), style,
                                      norm_mode, ctypes.cast(offs, ctypes.c_void_p), len(offsets),
                                      p_cur.data_ptr(), n_prompt, n_recent, scores.data_ptr(),
                                      _stream(stream)))
    return scores


def select_topk(scores: torch.Tensor, kv: KVCache, n_prompt: int, n_recent: int, budget: int,
                keep: torch.Tensor, stream=None) -> torch.Tensor:
    """Protected top-budget keep lists [S, budget] int32, ascending (tri_select_topk)."""
    lib = load_library()
    assert keep.dtype == torch.int32 and keep.is_contiguous() and keep.numel() == kv.n_slices * budget
    kvs = kv._abi()
    _check("tri_select_topk", lib.tri_select_topk(scores.data_ptr(), ctypes.byref(kvs), n_prompt,
                                                  n_recent, budget, keep.data_ptr(), _stream(stream)))
    return keep


def rand_evict(kv: KVCache, seed: int, rnd: int, n_prompt: int, n_recent: int, budget: int,
               keep: torch.Tensor, stream=None) -> torch.Tensor:
    """Random Attention keep lists [S, budget] int32 (rand_evict)."""
    lib = load_library()
    assert keep.dtype == torch.int32 and keep.is_contiguous() and keep.numel() == kv.n_slices * budget
    kvs = kv._abi()
    _check("rand_evict", lib.rand_evict(ctypes.byref(kvs), seed, rnd, n_prompt, n_recent, budget,
                                        keep.data_ptr(), _stream(stream)))
    return keep


DRAW_PER_HEAD, DRAW_PER_LAYER, DRAW_PER_SEQUENCE = 0, 1, 2


def rand_evict_scoped(kv: KVCache, seed: int, rnd: int, scope: int, n_prompt: int, n_recent: int, budget: int,
                      keep: torch.Tensor, stream=None) -> torch.Tensor:
    """Random Attention keep lists with the draw shared by every KV head of a
    layer (DRAW_PER_LAYER) or of a sequence (DRAW_PER_SEQUENCE) (rand_evict_scoped)."""
    lib = load_library()
    assert keep.dtype == torch.int32 and keep.is_contiguous() and keep.numel() == kv.n_slices * budget
    kvs = kv._abi()
    _check("rand_evict_scoped", lib.rand_evict_scoped(ctypes.byref(kvs), seed, rnd, scope, n_prompt, n_recent,
                                                      budget, keep.data_ptr(), _stream(stream)))
    return keep


def compact_kv(kv: KVCache, keep: torch.Tensor, budget: int, stream=None) -> None:
    """In-place order-preserving compaction of K, V and positions (tri_compact_kv)."""
    lib = load_library()
    assert keep.dtype == torch.int32 and keep.is_contiguous() and keep.numel() == kv.n_slices * budget
    kvs = kv._abi()
    _check("tri_compact_kv", lib.tri_compact_kv(ctypes.byref(kvs), keep.data_ptr(), budget,
                                                _stream(stream)))


def select_compact(scores: torch.Tensor, kv, n_prompt: int, n_recent: int, budget: int, keep: torch.Tensor,
                   stream=None) -> torch.Tensor:
    """select_topk then compact_kv, one kernel (tri_select_compact)."""
    lib = load_library()
    assert keep.dtype == torch.int32 and keep.is_contiguous() and keep.numel() == kv.n_slices * budget
    kvs = kv._abi()
    _check("tri_select_compact", lib.tri_select_compact(scores.data_ptr(), ctypes.byref(kvs), n_prompt, n_recent,
                                                        budget, keep.data_ptr(), _stream(stream)))
    return keep


def rand_evict_compact(kv, seed: int, rnd: int, n_prompt: int, n_recent: int, budget: int, keep: torch.Tensor,
                       scope: int = 0, stream=None) -> torch.Tensor:
    """rand_evict_scoped then compact_kv, one kernel (rand_evict_compact)."""
    lib = load_library()
    assert keep.dtype == torch.int32 and keep.is_contiguous() and keep.numel() == kv.n_slices * budget
    kvs = kv._abi()
    _check("rand_evict_compact", lib.rand_evict_compact(ctypes.byref(kvs), seed, rnd, scope, n_prompt, n_recent,
                                                        budget, keep.data_ptr(), _stream(stream)))
    return keep


def compress_workspace_bytes(kv: KVCache) -> int:
    kvs = kv._abi()
    return int(load_library().tri_compress_workspace_bytes(ctypes.byref(kvs)))


def compress(kv: KVCache, centers: Centers, rope_theta: float, offsets, p_cur: torch.Tensor,
             n_prompt: int, n_recent: int, budget: int, keep: torch.Tensor,
             workspace: torch.Tensor | None = None, style: int = ROPE_INTERLEAVED,
             norm_mode: int = NORM_WEIGHTED, stream=None) -> torch.Tensor:
    """One compression event: score + select + compact (tri_compress)."""
    lib = load_library()
    offs = (ctypes.c_int32 * len(offsets))(*[int(o) for o in offsets])
    assert p_cur.dtype == torch.int64 and p_cur.is_cuda
    assert keep.dtype == torch.int32 and keep.is_contiguous() and keep.numel() == kv.n_slices * budget
    kvs, cs = kv._abi(), centers._abi()
    need = int(lib.tri_compress_workspace_bytes(ctypes.byref(kvs)))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=kv.device)
    assert workspace.numel() >= need
    _check("tri_compress", lib.tri_compress(ctypes.byref(kvs), ctypes.byref(cs), float(rope_theta), style,
                                            norm_mode, ctypes.cast(offs, ctypes.c_void_p), len(offsets),
                                            p_cur.data_ptr(), n_prompt, n_recent, budget, keep.data_ptr(),
                                            workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return keep


def score_heads_workspace_bytes(kv: KVCache, group: int) -> int:
    kvs = kv._abi()
    return int(load_library().tri_score_heads_workspace_bytes(ctypes.byref(kvs), group))


def score_heads(kv: KVCache, centers: Centers, group: int, rope_theta: float, offsets, p_cur: torch.Tensor,
                scores_g: torch.Tensor, stats: torch.Tensor, workspace: torch.Tensor | None = None,
                style: int = ROPE_INTERLEAVED, norm_mode: int = NORM_WEIGHTED, stream=None):
    """Per-query-head scores [S, group, n_cap] of every valid row and their
    per-head (mean, std) [S, group, 2] (tri_score_heads). `centers` holds one
    row per query head (calibrate_centers with group=1)."""
    lib = load_library()
    offs = (ctypes.c_int32 * len(offsets))(*[int(o) for o in offsets])
    assert p_cur.dtype == torch.int64 and p_cur.is_cuda
    assert scores_g.dtype == torch.float32 and scores_g.is_contiguous()
    assert scores_g.numel() == kv.n_slices * group * kv.n_cap
    assert stats.dtype == torch.float32 and stats.is_contiguous() and stats.numel() == kv.n_slices * group * 2
    kvs, cs = kv._abi(), centers._abi()
    need = int(lib.tri_score_heads_workspace_bytes(ctypes.byref(kvs), group))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=kv.device)
    assert workspace.numel() >= need
    _check("tri_score_heads", lib.tri_score_heads(
        ctypes.byref(kvs), ctypes.byref(cs), group, float(rope_theta), style, norm_mode,
        ctypes.cast(offs, ctypes.c_void_p), len(offsets), p_cur.data_ptr(), scores_g.data_ptr(),
        stats.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return scores_g, stats


def select_topk_zmax(scores_g: torch.Tensor, stats: torch.Tensor, group: int, kv: KVCache, n_prompt: int,
                     n_recent: int, budget: int, keep: torch.Tensor, final_scores: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """Protected top-budget keep lists ranked by the GQA z-score maximum
    (tri_select_topk_zmax); optionally writes the final scores [S, n_cap]."""
    lib = load_library()
    assert keep.dtype == torch.int32 and keep.is_contiguous() and keep.numel() == kv.n_slices * budget
    if final_scores is not None:
        assert final_scores.dtype == torch.float32 and final_scores.is_contiguous()
        assert final_scores.numel() == kv.n_slices * kv.n_cap
    kvs = kv._abi()
    _check("tri_select_topk_zmax", lib.tri_select_topk_zmax(
        scores_g.data_ptr(), stats.data_ptr(), group, ctypes.byref(kvs), n_prompt, n_recent, budget,
        keep.data_ptr(), _ptr(final_scores), _stream(stream)))
    return keep


def select_union_workspace_bytes(kv: KVCache, n_prompt: int, n_recent: int, k_head: int) -> int:
    kvs = kv._abi()
    return int(load_library().tri_select_union_workspace_bytes(ctypes.byref(kvs), n_prompt, n_recent, k_head))


def select_union(scores: torch.Tensor, kv: KVCache, n_prompt: int, n_recent: int, budget: int, k_head: int,
                 keep: torch.Tensor, final_scores: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One keep list per (seq, layer) shared by its KV heads: union of every
    head's top k_head, ranked by the z-score maximum, topped up by it
    (tri_select_union). `scores` must cover every valid row."""
    lib = load_library()
    assert keep.dtype == torch.int32 and keep.is_contiguous() and keep.numel() == kv.n_slices * budget
    kvs = kv._abi()
    need = int(lib.tri_select_union_workspace_bytes(ctypes.byref(kvs), n_prompt, n_recent, k_head))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=kv.device)
    assert workspace.numel() >= need
    if final_scores is not None:
        assert final_scores.dtype == torch.float32 and final_scores.is_contiguous()
    _check("tri_select_union", lib.tri_select_union(
        scores.data_ptr(), ctypes.byref(kvs), n_prompt, n_recent, budget, k_head, keep.data_ptr(),
        _ptr(final_scores), workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return keep
