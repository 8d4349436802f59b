"""Seeded synthetic inputs for KV-cache scoring and compression.

This module only *makes data*: it draws Gaussian tensors from seeded torch
generators, applies rotary position embedding (RoPE) to queries and keys,
scales a few outlier key channels and writes attention-sink keys.  It holds
none of the method's arithmetic (no attention scores, weights, allocation or
quantisation), so both the CUDA path and the CPU oracle may consume it.

Shapes (row-major, contiguous):
    Q    [Hq,  W, d]   queries of the observation window, positions q_pos0 .. q_pos0+W-1
    K, V [Hkv, N, d]   the prefilled cache, positions 0 .. N-1
    h    [W, D]        hidden states of the query positions (KVzip+ only)
    W_O  [D, Hq*d]     output projection (KVzip+ only)

The workloads stand in for the model activations that the RDKV and KVzap
papers evaluate on (LLaMA / Mistral / Qwen layers over LongBench, RULER,
InfiniteBench): none of those weights or datasets is available, so
Llama-3-8B-shaped Gaussian tensors with RoPE, outlier channels and sink keys
are used instead.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

# tensor ids used in the seed formula
_TID = {"Q": 1, "K": 2, "V": 3, "h": 4, "h_scale": 5, "W_O": 6, "outlier_perm": 7}


def seed_of(family: int, layer: int, seq: int, tensor: str) -> int:
    """s = 1_000_003*family + 1009*layer + 97*seq + tensor_id."""
    return 1_000_003 * family + 1009 * layer + 97 * seq + _TID[tensor]


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: sizes, the distribution knobs and the budgets."""
    name: str
    family: int                  # seed family id
    Hq: int
    Hkv: int
    N: int                       # keys / values per sequence
    W: int                       # observation-window queries (last W positions)
    d: int
    D: int = 0                   # hidden size (KVzip+ only)
    layers: int = 1
    seqs: int = 1
    outlier_channels: int = 0
    outlier_scale: float = 1.0   # constant scale, or see outlier_scale_of()
    layer_dependent_outliers: bool = False
    n_sinks: int = 0
    mode: str = "rdkv"           # "rdkv" or "kvzip_plus"
    avg_bits: tuple = (4,)       # average bits per unit (budget sweep)
    widths: tuple = (0, 2, 4, 8, 16)
    evict_fraction: float = 0.0  # kvzip_plus: fraction of units evicted (widths {0,16})
    extra: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def q_pos0(self) -> int:
        return self.N - self.W

    def small(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # single head causal prefill, every position is a query
    "single_head_n512_d64": Workload(
        name="single_head_n512_d64", family=1, Hq=1, Hkv=1, N=512, W=512, d=64,
        avg_bits=(4,)),
    # Llama-3-8B-shaped layer: 32 q heads, 8 kv heads, window 512 of 8192
    "llama3_8b_layer_n8192_w512": Workload(
        name="llama3_8b_layer_n8192_w512", family=2, Hq=32, Hkv=8, N=8192, W=512,
        d=128, outlier_channels=4, outlier_scale=8.0, n_sinks=4, avg_bits=(3,)),
    # KVzip+ over a repeated prompt: full N x N causal, hidden 4096
    "kvzip_plus_n32768_d4096": Workload(
        name="kvzip_plus_n32768_d4096", family=3, Hq=32, Hkv=8, N=32768, W=32768,
        d=128, D=4096, mode="kvzip_plus", widths=(0, 16), evict_fraction=0.8),
    # long-context layer: window 4096 of 131072, 16 sinks, budgets 2/3/4
    "long_context_n131072_w4096": Workload(
        name="long_context_n131072_w4096", family=4, Hq=32, Hkv=8, N=131072, W=4096,
        d=128, outlier_channels=4, outlier_scale=8.0, n_sinks=16, avg_bits=(2, 3, 4)),
    # full model: 32 layers x 16 sequences x 16384 tokens, window 1024
    "full_model_l32_b16_n16384": Workload(
        name="full_model_l32_b16_n16384", family=5, Hq=32, Hkv=8, N=16384, W=1024,
        d=128, layers=32, seqs=16, outlier_channels=4, layer_dependent_outliers=True,
        n_sinks=4, avg_bits=(3,)),
}


def outlier_scale_of(wl: Workload, layer: int) -> float:
    if wl.layer_dependent_outliers:
        return 2.0 + 8.0 * layer / max(wl.layers - 1, 1)
    return wl.outlier_scale


def _normal(shape, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def apply_rope(x: torch.Tensor, pos: torch.Tensor) -> torch.Tensor:
    """Rotate-half RoPE with base 10000: pairs (c, c + d/2), angle pos * 10000^(-2i/d)."""
    d = x.shape[-1]
    half = d // 2
    inv = torch.pow(torch.tensor(10000.0, dtype=torch.float64, device=x.device),
                    -torch.arange(half, dtype=torch.float64, device=x.device) * 2.0 / d)
    ang = pos.to(torch.float64)[:, None] * inv[None, :]
    cos = torch.cos(ang).to(torch.float32)
    sin = torch.sin(ang).to(torch.float32)
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def make_layer(wl: Workload, layer: int = 0, seq: int = 0, device="cpu") -> dict:
    """Q, K, V (bf16) for one (layer, sequence) of a workload.

    Order: N(0,1) fp32 -> RoPE -> outlier channels -> sink keys -> bf16.
    Sink keys are 3*sqrt(d) times the unit vector of the mean post-RoPE window
    query of the KV group's heads (a key of typical length sqrt(d) pointing
    where the queries point, scaled 3x).
    """
    f, dev = wl.family, torch.device(device)
    Q = _normal((wl.Hq, wl.W, wl.d), seed_of(f, layer, seq, "Q"), dev)
    K = _normal((wl.Hkv, wl.N, wl.d), seed_of(f, layer, seq, "K"), dev)
    V = _normal((wl.Hkv, wl.N, wl.d), seed_of(f, layer, seq, "V"), dev)
    qpos = torch.arange(wl.q_pos0, wl.q_pos0 + wl.W, device=dev)
    kpos = torch.arange(wl.N, device=dev)
    Q = apply_rope(Q, qpos)
    K = apply_rope(K, kpos)
    if wl.outlier_channels:
        g = torch.Generator(device="cpu")
        g.manual_seed(seed_of(f, layer, seq, "outlier_perm"))
        chans = torch.randperm(wl.d, generator=g)[: wl.outlier_channels].to(dev)
        K[:, :, chans] *= outlier_scale_of(wl, layer)
    if wl.n_sinks:
        G = wl.G
        for gi in range(wl.Hkv):
            mq = Q[gi * G:(gi + 1) * G].reshape(-1, wl.d).mean(dim=0)
            u = mq / mq.norm().clamp_min(1e-30)
            K[gi, : wl.n_sinks, :] = 3.0 * math.sqrt(wl.d) * u
    out = {"Q": Q.to(torch.bfloat16).contiguous(),
           "K": K.to(torch.bfloat16).contiguous(),
           "V": V.to(torch.bfloat16).contiguous()}
    if wl.mode == "kvzip_plus":
        z = _normal((wl.W, wl.D), seed_of(f, layer, seq, "h"), dev)
        eps = _normal((wl.W,), seed_of(f, layer, seq, "h_scale"), dev)
        out["h"] = (z * torch.exp(0.5 * eps)[:, None]).to(torch.bfloat16).contiguous()
        wo = _normal((wl.D, wl.Hq * wl.d), seed_of(f, layer, seq, "W_O"), dev)
        out["W_O"] = (wo / math.sqrt(wl.D)).to(torch.bfloat16).contiguous()
    return out


def make_pools(wl: Workload, layer: int, seqs, device="cpu") -> dict:
    """Q [P*Hq, W, d], K and V [P*Hkv, N, d] (bf16) of the sequences `seqs` of one
    layer, stacked pool after pool (pool i = sequence seqs[i], made by make_layer).
    On a CUDA device the Gaussians come from that device's generator."""
    seqs = list(seqs)
    P = len(seqs)
    dev = torch.device(device)
    out = {"Q": torch.empty(P * wl.Hq, wl.W, wl.d, dtype=torch.bfloat16, device=dev),
           "K": torch.empty(P * wl.Hkv, wl.N, wl.d, dtype=torch.bfloat16, device=dev),
           "V": torch.empty(P * wl.Hkv, wl.N, wl.d, dtype=torch.bfloat16, device=dev)}
    for i, sq in enumerate(seqs):
        t = make_layer(wl, layer, sq, device=dev)
        out["Q"][i * wl.Hq:(i + 1) * wl.Hq] = t["Q"]
        out["K"][i * wl.Hkv:(i + 1) * wl.Hkv] = t["K"]
        out["V"][i * wl.Hkv:(i + 1) * wl.Hkv] = t["V"]
    return out


def budget_bits(avg_bits: float, units: int) -> int:
    """Total budget B = floor(avg_bits * U) bits (widths counted per unit)."""
    return int(math.floor(avg_bits * units))


def kvzip_keep_budget(U: int, evict_fraction: float) -> int:
    """Widths {0,16}: keep U - floor(f*U) units at 16 bits -> B = 16*keep."""
    keep = U - int(math.floor(evict_fraction * U))
    return 16 * keep
