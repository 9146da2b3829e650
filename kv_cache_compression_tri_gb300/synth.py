"""Seeded synthetic inputs shaped like the pages' long-reasoning workloads.

This module only draws random numbers (torch generators, seeded) and lays
them out; it contains none of the compression arithmetic, so both the CUDA
path and the oracle can consume what it makes.

Recipe (all draws from one torch.Generator per workload, seed 0 unless
stated, in this order):
  1. key centres  mu_k[layer, kv_head, :]  ~ N(0, 1) per dim, rescaled to
     norm `key_center_norm`;
  2. query centres mu_q[layer, q_head, :]  the same, norm `q_center_norm`;
  3. calibration queries q[layer, q_head, t, :] = mu_q + q_noise_std * N(0, 1),
     n_cal rows per query head;
  4. keys k[seq, layer, head, i, :] = mu_k[layer, head] + key_noise_std * N(0, 1)
     and values v ~ value_std * N(0, 1), drawn (seq, layer) by (seq, layer)
     in fp32 and rounded once to the cache dtype.
Rows appended by the periodic workload in round r come from a generator
seeded with (seed * 1_000_003 + 1 + r) and follow step 4.

Workloads with key_layout "post" store what an engine stores: each key row
rotated by the model's RoPE at its slot position (rope_rows below; RoPE is
the model's position encoding, not part of the compression method), drawn
in fp32 and rounded once to the cache dtype.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n_seq: int
    n_layers: int
    n_kv_heads: int
    group: int  # query heads per KV head
    head_dim: int
    theta: float
    dtype: torch.dtype
    n_cap: int
    n_valid: int
    n_prompt: int
    n_recent: int
    budget: int
    offsets: tuple = ()
    key_center_norm: float = 8.0
    key_noise_std: float = 1.0
    value_std: float = 1.0
    q_center_norm: float = 8.0
    q_noise_std: float = 1.0
    n_cal: int = 4096
    random: bool = False  # Random Attention variant (no centres, no score)
    rounds: int = 0  # periodic rounds after the first compression
    round_rows: int = 0
    seed: int = 0
    key_layout: str = "pre"  # "post": keys stored RoPE-rotated at their slot positions
    description: str = ""

    @property
    def n_slices(self) -> int:
        return self.n_seq * self.n_layers * self.n_kv_heads

    @property
    def n_q_heads(self) -> int:
        return self.n_kv_heads * self.group

    @property
    def elem_bytes(self) -> int:
        return torch.tensor([], dtype=self.dtype).element_size()


def _geo(lo_exp: int, hi_exp: int) -> tuple:
    return tuple(2 ** j for j in range(lo_exp, hi_exp + 1))


WORKLOADS = {
    "tiny": Workload(
        "tiny", n_seq=1, n_layers=1, n_kv_heads=2, group=1, head_dim=64, theta=1e4,
        dtype=torch.float32, n_cap=512, n_valid=512, n_prompt=32, n_recent=64, budget=128,
        offsets=_geo(0, 10), description="1 layer x 2 KV heads, d 64, fp32, 512 tokens -> 128"),
    "qwen3_8b_layer": Workload(
        "qwen3_8b_layer", n_seq=1, n_layers=1, n_kv_heads=8, group=4, head_dim=128, theta=1e6,
        dtype=torch.bfloat16, n_cap=2176, n_valid=2176, n_prompt=256, n_recent=128, budget=2048,
        offsets=_geo(0, 14), key_center_norm=12.0, key_noise_std=1.5, q_center_norm=12.0,
        q_noise_std=1.5, description="Qwen3-8B-shaped layer: 8 KV heads (GQA 4), d 128, bf16, 2176 -> 2048"),
    "qwen3_8b_stack": Workload(
        "qwen3_8b_stack", n_seq=16, n_layers=36, n_kv_heads=8, group=4, head_dim=128, theta=1e6,
        dtype=torch.bfloat16, n_cap=32768, n_valid=32768, n_prompt=512, n_recent=128, budget=4096,
        offsets=_geo(0, 16),
        description="Qwen3-8B-shaped stack: 16 seqs x 36 layers x 8 KV heads, d 128, bf16, 32768 -> 4096"),
    "random_stack": Workload(
        "random_stack", n_seq=16, n_layers=36, n_kv_heads=8, group=4, head_dim=128, theta=1e6,
        dtype=torch.bfloat16, n_cap=32768, n_valid=32768, n_prompt=512, n_recent=0, budget=4096,
        random=True, description="Random Attention on the 16 x 36 x 8 stack, prompt 512, 32768 -> 4096"),
    "periodic_large_batch": Workload(
        "periodic_large_batch", n_seq=64, n_layers=24, n_kv_heads=8, group=1, head_dim=64,
        theta=1.5e5, dtype=torch.bfloat16, n_cap=32768, n_valid=32768, n_prompt=1024,
        n_recent=128, budget=2048, offsets=_geo(0, 16), rounds=16, round_rows=128,
        description="64 seqs x 24 layers x 8 KV heads, d 64, bf16, 32768 -> 2048 then 16 rounds of +128"),
}

# The five workloads in the order the task lists them (1-based numbering).
BY_NUMBER = {1: "tiny", 2: "qwen3_8b_layer", 3: "qwen3_8b_stack", 4: "random_stack",
             5: "periodic_large_batch"}


def scaled(w: Workload, **over) -> Workload:
    """A copy of a workload with some fields replaced (smaller test cases)."""
    d = {f: getattr(w, f) for f in w.__dataclass_fields__}
    d.update(over)
    return Workload(**d)


# Profiling case: the stack with one sequence (288 slices, 2.4 GB of K).
WORKLOADS["qwen3_8b_stack_1seq"] = scaled(WORKLOADS["qwen3_8b_stack"], name="qwen3_8b_stack_1seq", n_seq=1,
                                          description="one sequence of the Qwen3-8B-shaped stack")
WORKLOADS["random_stack_1seq"] = scaled(WORKLOADS["random_stack"], name="random_stack_1seq", n_seq=1,
                                        description="one sequence of the Random Attention stack")
WORKLOADS["qwen3_8b_stack_post_rope"] = scaled(
    WORKLOADS["qwen3_8b_stack"], name="qwen3_8b_stack_post_rope", key_layout="post",
    description="the Qwen3-8B-shaped stack with keys stored post-RoPE, as engines keep them")
WORKLOADS["qwen3_8b_stack_post_rope_1seq"] = scaled(
    WORKLOADS["qwen3_8b_stack_post_rope"], name="qwen3_8b_stack_post_rope_1seq", n_seq=1,
    description="one sequence of the post-RoPE stack")
WORKLOADS["periodic_1seq"] = scaled(WORKLOADS["periodic_large_batch"], name="periodic_1seq", n_seq=1,
                                    description="one sequence of the large-batch periodic workload")
# Profiling case for the periodic rounds' shape (2176 rows -> 2048, one
# score CTA per slice): four sequences, 0.43 GB of K and V (more than L2).
WORKLOADS["periodic_round_4seq"] = scaled(WORKLOADS["periodic_large_batch"], name="periodic_round_4seq", n_seq=4,
                                          n_cap=2176, n_valid=2176, rounds=0,
                                          description="four sequences of a periodic round: 2176 rows -> 2048")


def _unit_rows(g: torch.Generator, shape, norm: float, device) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return x * (norm / x.norm(dim=-1, keepdim=True))


def rope_rows(x: torch.Tensor, pos: torch.Tensor, theta: float, style: int = 0) -> torch.Tensor:
    """The model's RoPE of rows x [..., n, d] at positions pos [n]: band f --
    (x[2f], x[2f+1]) for style 0, (x[f], x[f+d/2]) for style 1 -- rotated by
    angle theta^(-2f/d) * pos. Angles in fp64, result in fp32."""
    d = x.shape[-1]
    F = d // 2
    f = torch.arange(F, dtype=torch.float64, device=x.device)
    omega = torch.pow(torch.tensor(float(theta), dtype=torch.float64, device=x.device), -2.0 * f / d)
    ang = pos.to(torch.float64)[:, None] * omega[None, :]
    cs, sn = torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)
    x = x.to(torch.float32)
    if style == 0:
        a, b = x[..., 0::2], x[..., 1::2]
    else:
        a, b = x[..., :F], x[..., F:]
    ra, rb = a * cs - b * sn, a * sn + b * cs
    out = torch.empty_like(x)
    if style == 0:
        out[..., 0::2], out[..., 1::2] = ra, rb
    else:
        out[..., :F], out[..., F:] = ra, rb
    return out


@dataclass
class Inputs:
    w: Workload
    mu_k: torch.Tensor  # [L, H, d] fp32
    mu_q: torch.Tensor  # [L, Hq, d] fp32
    q: torch.Tensor | None  # [L, Hq, n_cal, d] in w.dtype
    k: torch.Tensor  # [n_seq, L, H, n_cap, d]
    v: torch.Tensor
    n_valid: torch.Tensor  # [S] int32
    p_cur: torch.Tensor  # [n_seq] int64
    extra: dict = field(default_factory=dict)


def make_inputs(w: Workload, device="cuda", with_queries: bool = True, seqs: int | None = None) -> Inputs:
    """Draw the workload's centres, calibration queries and cache.
    `seqs` limits the number of sequences drawn (the first ones)."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    L, H, Hq, d = w.n_layers, w.n_kv_heads, w.n_q_heads, w.head_dim
    mu_k = _unit_rows(g, (L, H, d), w.key_center_norm, device)
    mu_q = _unit_rows(g, (L, Hq, d), w.q_center_norm, device)
    q = None
    if with_queries and not w.random:
        q = torch.empty(L, Hq, w.n_cal, d, dtype=w.dtype, device=device)
        for l in range(L):
            noise = torch.randn(Hq, w.n_cal, d, generator=g, device=device)
            q[l] = (mu_q[l][:, None, :] + w.q_noise_std * noise).to(w.dtype)
    n_seq = w.n_seq if seqs is None else min(seqs, w.n_seq)
    k = torch.empty(n_seq, L, H, w.n_cap, d, dtype=w.dtype, device=device)
    v = torch.empty_like(k)
    rows = w.n_valid
    slots = torch.arange(rows, device=device)
    for s in range(n_seq):
        for l in range(L):
            noise = torch.randn(H, rows, d, generator=g, device=device)
            kk = mu_k[l][:, None, :] + w.key_noise_std * noise
            if w.key_layout == "post":
                kk = rope_rows(kk, slots, w.theta)
            k[s, l, :, :rows] = kk.to(w.dtype)
            v[s, l, :, :rows] = (w.value_std * torch.randn(H, rows, d, generator=g, device=device)).to(w.dtype)
            if rows < w.n_cap:
                k[s, l, :, rows:] = 0
                v[s, l, :, rows:] = 0
    n_valid = torch.full((n_seq * L * H,), rows, dtype=torch.int32, device=device)
    p_cur = torch.full((n_seq,), rows - 1, dtype=torch.int64, device=device)
    return Inputs(w, mu_k, mu_q, q, k, v, n_valid, p_cur)


def append_rows(inp: Inputs, rnd: int, n_rows: int, device=None):
    """Fresh K/V rows of periodic round `rnd` (>= 1): [n_seq, L, H, n_rows, d]."""
    w = inp.w
    device = torch.device(device) if device is not None else inp.k.device
    g = torch.Generator(device=device)
    g.manual_seed(w.seed * 1_000_003 + 1 + rnd)
    n_seq, L, H, _, d = inp.k.shape
    kn = torch.empty(n_seq, L, H, n_rows, d, dtype=w.dtype, device=device)
    vn = torch.empty_like(kn)
    mu = inp.mu_k.to(device)
    for s in range(n_seq):
        for l in range(L):
            noise = torch.randn(H, n_rows, d, generator=g, device=device)
            kn[s, l] = (mu[l][:, None, :] + w.key_noise_std * noise).to(w.dtype)
            vn[s, l] = (w.value_std * torch.randn(H, n_rows, d, generator=g, device=device)).to(w.dtype)
    return kn, vn


def sample_slices(n_slices: int, count: int = 48) -> list[int]:
    """Deterministic slice sample: first, last and evenly strided between."""
    if n_slices <= count:
        return list(range(n_slices))
    idx = {0, n_slices - 1}
    for j in range(1, count - 1):
        idx.add((j * (n_slices - 1)) // (count - 1))
    return sorted(idx)


def kv_cache_bytes(layers: int, d_model: int, tokens: int, elem_bytes: int, batch: int = 1) -> int:
    """Bytes of a K+V cache: batch x 2 x layers x d_model x tokens x elem_bytes
    (d_model = heads x head_dim)."""
    return batch * 2 * layers * d_model * tokens * elem_bytes
