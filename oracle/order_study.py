"""Order study of the OScaR key path on synthetic sinks (float64, CPU).

TEST INFRASTRUCTURE ONLY, like the oracle it calls: the test-suite runs it,
and ``python -m oracle.order_study`` prints its report.  Nothing in the
library calls it.

The pages motivate the method's two key-side stages by their effect on keys
(ai-papers.net summary of OScaR, section "OScaRの提案手法"): the Hadamard
rotation spreads channel-outlier energy over all dimensions, the per-token
norm scaling equalises token norms, and the rotation has to come first.  The
OScaR abstract (arXiv 2605.19660) names the failure it addresses on the
token side: small-norm tokens, such as attention sinks, crushed by a
per-channel quantiser whose step is set by the large-norm tokens.

This harness quantises the same synthetic keys through five key pipelines
and reports, per pipeline:

* the relative reconstruction error ||k_hat - k|| / ||k|| of ordinary tokens
  and of sink tokens (norm <= 0.1 x the head's median norm);
* the error of the attention output against exact float64 attention, with
  the values left exact so that only the key path differs.

Pipelines (all per-channel asymmetric INT2 over 128-token groups, as in the
oracle):

* ``rotate_then_scale``: the method (Canalized Rotation, then Omni-Token
  Scaling);
* ``scale_then_rotate``: the reversed order;
* ``rotate_only``: no per-token scaling;
* ``scale_only``: no rotation;
* ``per_channel_only``: neither (per-channel keys as in KIVI).
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from . import oscar_oracle as O

VARIANTS: Dict[str, dict] = {
    "rotate_then_scale": dict(rotate=True, scale=True, scale_first=False),
    "scale_then_rotate": dict(rotate=True, scale=True, scale_first=True),
    "rotate_only": dict(rotate=True, scale=False),
    "scale_only": dict(rotate=False, scale=True),
    "per_channel_only": dict(rotate=False, scale=False),
}

SINK_NORM_RATIO = 0.1   # a token is a sink if its norm is <= this x the head's median norm


def dequantised_keys(k: np.ndarray, variant: str) -> np.ndarray:
    """Keys of one head [L, d] (L a multiple of the group size) after the
    given pipeline and back, in the original basis and scale."""
    k = np.asarray(k, dtype=np.float64)
    L, d = k.shape
    g = k.reshape(L // O.KEY_GROUP, O.KEY_GROUP, d)
    return O.quantize_key_group_variant(g, **VARIANTS[variant]).reshape(L, d)


def sink_mask(k: np.ndarray) -> np.ndarray:
    n = np.linalg.norm(np.asarray(k, dtype=np.float64), axis=-1)
    return n <= SINK_NORM_RATIO * np.median(n)


def key_errors(k: np.ndarray, kh: np.ndarray, sinks: np.ndarray) -> dict:
    n = np.linalg.norm(k, axis=-1)
    rel = np.linalg.norm(kh - k, axis=-1) / np.where(n > 0, n, 1.0)
    out = {"key_rel_err": float(rel[~sinks].mean())}
    if sinks.any():
        out["sink_key_rel_err"] = float(rel[sinks].mean())
        out["sink_key_rel_err_max"] = float(rel[sinks].max())
    return out


def attention_error(q: np.ndarray, k: np.ndarray, kh: np.ndarray, v: np.ndarray) -> dict:
    """Max / mean |o - o_exact| for queries q [h, d] against one head's
    dequantised keys kh, with the exact values v [L, d] on both sides."""
    o_ref = O.attention_exact(q, k, v)
    o = O.attention_exact(q, kh, v)
    e = np.abs(o - o_ref)
    return {"attn_max_abs_err": float(e.max()), "attn_mean_abs_err": float(e.mean())}


def study(L: int = 4096, hkv: int = 2, gqa: int = 4, seed: int = 4,
          variants: Optional[list] = None) -> Dict[str, dict]:
    """Run every pipeline on a seeded synthetic layer (Llama-layer recipe with
    1% random sinks besides token 0) and return the per-pipeline report,
    averaged over KV heads (maxima taken over heads)."""
    import torch

    from int2_kv_cache_oscar_gb300 import workloads as W

    r = W.KVRecipe(k_outliers_per_head=4, k_outlier_scale=15.0, lognormal_sigma=0.5, sink_token0=True,
                   sink_fraction=0.01, v_outliers_per_head=2, v_outlier_scale=5.0)
    gen = torch.Generator().manual_seed(seed)
    k, v = W.make_sequence_kv(L, hkv, r, gen)
    q = W.make_q(1, hkv * gqa, seed=seed + 1)[0]
    kf = k.float().numpy().astype(np.float64)
    vf = v.float().numpy().astype(np.float64)
    qf = q.float().numpy().astype(np.float64)
    report: Dict[str, dict] = {}
    for name in (variants or list(VARIANTS)):
        acc: Dict[str, list] = {}
        for j in range(hkv):
            kj, vj = kf[:, j], vf[:, j]
            sinks = sink_mask(kj)
            kh = dequantised_keys(kj, name)
            res = key_errors(kj, kh, sinks)
            res.update(attention_error(qf[j * gqa:(j + 1) * gqa], kj, kh, vj))
            res["n_sinks"] = int(sinks.sum())
            for key, val in res.items():
                acc.setdefault(key, []).append(val)
        report[name] = {key: (float(np.max(vals)) if key.endswith("max") or key.startswith("attn_max")
                              else float(np.sum(vals)) if key == "n_sinks" else float(np.mean(vals)))
                        for key, vals in acc.items()}
    return report


def format_report(report: Dict[str, dict]) -> str:
    cols = ["key_rel_err", "sink_key_rel_err", "sink_key_rel_err_max", "attn_max_abs_err", "attn_mean_abs_err"]
    lines = ["| pipeline | " + " | ".join(cols) + " |", "|---" * (len(cols) + 1) + "|"]
    for name, r in report.items():
        lines.append(f"| {name} | " + " | ".join(f"{r.get(c, float('nan')):.4g}" for c in cols) + " |")
    return "\n".join(lines)


if __name__ == "__main__":
    import sys

    L = int(sys.argv[1]) if len(sys.argv) > 1 else 4096
    rep = study(L=L)
    n = next(iter(rep.values()))["n_sinks"]
    print(f"order study: L={L}, 2 KV heads x 4 query heads, seed 4, {n:.0f} sink tokens")
    print(format_report(rep))
