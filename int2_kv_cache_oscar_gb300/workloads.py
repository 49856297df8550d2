"""Seeded synthetic K/V/q generators for the OScaR INT2 KV-cache workloads.

This module only draws random tensors with the shapes and value structure of
the workloads the OScaR pages measure on (Llama-3.1-8B / Qwen3-8B layers at
8K-128K context, "OScaR: The Occam's Razor for Extreme KV Cache
Quantization", abstract; ai-papers.net summary, section "実験結果").  It holds
none of the method's arithmetic: no rotation, no norm division, no
quantisation.  Both the CUDA path and the CPU oracle receive the tensors it
returns, so neither side needs a generator of its own.

Recipe (every workload):
  * K ~ N(0, 1) fp32 [L, Hkv, d].  Per KV head, a set of "outlier" channels
    is multiplied by a factor (channel-wise outliers of keys).
  * Optionally every token's key is multiplied by exp(sigma * z), z ~ N(0,1)
    (lognormal token norms).
  * Sink tokens keep their direction; their L2 norm is set to
    ``sink_factor`` x the median token norm of that head (median taken after
    the outlier and lognormal scaling).  This is the token-norm imbalance
    (small-norm attention sinks) the OScaR pages describe.
  * V ~ N(0, 1) fp32 with a few channels per head multiplied by a factor.
  * q ~ N(0, 1) fp32 [B, Hq, d].
  * Everything is rounded to bf16 (round-to-nearest-even) at the end.

Draw order for one sequence: K, V, then the per-head outlier channel choices,
lognormal factors, sink positions; q is drawn after all sequences.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

HEAD_DIM = 128


@dataclass
class KVRecipe:
    """Value-structure recipe of one synthetic workload."""

    k_outlier_channels: Optional[Sequence[int]] = None  # fixed channels (all heads)
    k_outliers_per_head: int = 0                       # random channels per head
    k_outlier_scale: float = 1.0
    lognormal_sigma: float = 0.0
    sink_token0: bool = True
    sink_fraction: float = 0.0                          # extra random sinks
    sink_factor: float = 0.05
    v_outliers_per_head: int = 0
    v_outlier_scale: float = 1.0


@dataclass
class Workload:
    """A named workload: batch of sequences sharing one head layout."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    seq_lens: List[int]
    seed: int
    recipe: KVRecipe = field(default_factory=KVRecipe)
    head_dim: int = HEAD_DIM


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_sequence_kv(L: int, Hkv: int, recipe: KVRecipe, gen: torch.Generator,
                     device="cpu", d: int = HEAD_DIM):
    """Draw one sequence's K and V as bf16 tensors of shape [L, Hkv, d]."""
    k = torch.randn((L, Hkv, d), generator=gen, device=device, dtype=torch.float32)
    v = torch.randn((L, Hkv, d), generator=gen, device=device, dtype=torch.float32)
    if L == 0:
        return k.to(torch.bfloat16), v.to(torch.bfloat16)
    # channel outliers of K, per KV head
    for h in range(Hkv):
        if recipe.k_outlier_channels is not None:
            ch = torch.tensor(list(recipe.k_outlier_channels), device=device)
        elif recipe.k_outliers_per_head > 0:
            ch = torch.randperm(d, generator=gen, device=device)[: recipe.k_outliers_per_head]
        else:
            ch = None
        if ch is not None:
            k[:, h, ch] *= recipe.k_outlier_scale
        if recipe.v_outliers_per_head > 0:
            vch = torch.randperm(d, generator=gen, device=device)[: recipe.v_outliers_per_head]
            v[:, h, vch] *= recipe.v_outlier_scale
    if recipe.lognormal_sigma > 0.0:
        z = torch.randn((L, Hkv, 1), generator=gen, device=device, dtype=torch.float32)
        k *= torch.exp(recipe.lognormal_sigma * z)
    # sinks: keep direction, set norm to sink_factor x median norm of the head
    sinks = []
    if recipe.sink_token0:
        sinks.append(torch.zeros(1, dtype=torch.long, device=device))
    if recipe.sink_fraction > 0.0:
        n_extra = int(round(recipe.sink_fraction * L))
        if n_extra > 0:
            sinks.append(torch.randperm(L, generator=gen, device=device)[:n_extra])
    if sinks:
        pos = torch.unique(torch.cat(sinks))
        norms = torch.linalg.vector_norm(k, dim=-1)          # [L, Hkv]
        med = norms.median(dim=0).values                      # [Hkv]
        target = recipe.sink_factor * med                     # [Hkv]
        cur = norms[pos]                                      # [S, Hkv]
        k[pos] *= (target[None, :] / cur.clamp_min(1e-30))[..., None]
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def make_workload_tensors(w: Workload, device="cpu"):
    """Return (ks, vs, q): lists of per-sequence bf16 [L_b, Hkv, d] tensors and
    a bf16 q of shape [B, Hq, d]."""
    gen = _gen(w.seed, device)
    ks, vs = [], []
    for L in w.seq_lens:
        k, v = make_sequence_kv(L, w.num_kv_heads, w.recipe, gen, device, w.head_dim)
        ks.append(k)
        vs.append(v)
    q = torch.randn((w.batch, w.num_q_heads, w.head_dim), generator=gen,
                    device=device, dtype=torch.float32).to(torch.bfloat16)
    return ks, vs, q


def make_q(batch: int, Hq: int, seed: int, device="cpu", d: int = HEAD_DIM):
    gen = _gen(seed, device)
    return torch.randn((batch, Hq, d), generator=gen, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


LLAMA_RECIPE = KVRecipe(k_outliers_per_head=4, k_outlier_scale=15.0, lognormal_sigma=0.5,
                        sink_token0=True, v_outliers_per_head=2, v_outlier_scale=5.0)


def tiny_layer(L: int = 1024) -> Workload:
    """1 KV head, 4 query heads, d=128; K channels 3 and 77 x20; token-0 sink."""
    r = KVRecipe(k_outlier_channels=(3, 77), k_outlier_scale=20.0, sink_token0=True)
    return Workload("tiny-1kv-4q-L1024", 1, 4, 1, [L], seed=0, recipe=r)


def llama_layer(L: int = 8192, seed: int = 1) -> Workload:
    """Llama-3.1-8B-shaped layer: 32 query / 8 KV heads, d=128, batch 1."""
    return Workload(f"llama8b-layer-B1-L{L}", 1, 32, 8, [L], seed=seed, recipe=LLAMA_RECIPE)


def context_sweep(L: int) -> Workload:
    """Single-batch context sweep point (8K..128K) with the Llama layer recipe."""
    return Workload(f"sweep-B1-L{L}", 1, 32, 8, [L], seed=2, recipe=LLAMA_RECIPE)


def multi_batch(batch: int = 32, L: int = 32768) -> Workload:
    """Batch of equal-length sequences; sinks at token 0 plus 1% random positions."""
    r = KVRecipe(k_outliers_per_head=4, k_outlier_scale=15.0, lognormal_sigma=0.5,
                 sink_token0=True, sink_fraction=0.01, v_outliers_per_head=2,
                 v_outlier_scale=5.0)
    return Workload(f"multibatch-B{batch}-L{L}", batch, 32, 8, [L] * batch, seed=3, recipe=r)


def ragged_lengths(batch: int = 8, lo: int = 4096, hi: int = 131072, seed: int = 4) -> List[int]:
    gen = _gen(seed, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (batch,), generator=gen)]


def ragged_stream(batch: int = 8, lo: int = 4096, hi: int = 131072) -> Workload:
    """Ragged serving stream: lengths drawn uniformly from [lo, hi]."""
    return Workload(f"ragged-B{batch}", batch, 32, 8, ragged_lengths(batch, lo, hi), seed=4,
                    recipe=LLAMA_RECIPE)
