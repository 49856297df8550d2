"""CPU oracle for the OScaR INT2 KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and
the benchmark's CPU-baseline leg may import this module.  The library's
product path never calls it; it shares no code, tables or constants with the
CUDA kernels.

It is a plain, slow, obviously-correct restatement of the method in float64
numpy.  Sources:

* "OScaR: The Occam's Razor for Extreme KV Cache Quantization in LLMs and
  Beyond" (arXiv 2605.19660), Abstract: per-channel Key quantisation is kept,
  "Canalized Rotation followed by Omni-Token Scaling" is applied before it,
  and the cache is quantised to INT2.
* ai-papers.net summary of OScaR, section "OScaRの提案手法": stage 1 applies a
  Hadamard transform to spread channel-outlier energy over all dimensions;
  stage 2 computes every token's L2 norm and scales tokens to equalise norms;
  rotation must come first.
* qiita.com article on NOVA-KV, section "KV キャッシュを「読む」時間が、
  計算そのものより長い": the KIVI convention of quantising Keys per channel and
  Values per token (asymmetric rounding).

Readings taken where the pages are silent (each is also listed in the design
notes of the repository):

* H_d is the Sylvester-ordered Walsh-Hadamard matrix, normalised:
  H[i, j] = (-1)^popcount(i & j) / sqrt(d).  No random signs.
* Only keys are rotated; the query is rotated at decode time so that
  q_rot . k_rot = q . k.  Values are not rotated.
* The stored norm is the L2 norm of the rotated key (equal to that of the raw
  key); the key is divided by it; a zero-norm key becomes the zero vector.
* Asymmetric INT2: over the quantisation group, s = (max - min) / 3 and
  z = min, computed in float64 and stored as float32; code =
  clamp(round_half_even((x - z) / s), 0, 3) with (x - z) / s evaluated in
  float64 from the exact values of the stored parameters, so that the
  decision is the one the stored scale and zero define (an exact tie goes
  to the even code; a value a hair below a tie goes down even where a float32
  evaluation would round it onto the tie); s == 0 gives code 0 (dequantised
  value z).  Dequantised value = code * s + z.
* Keys: per channel over groups of G = 128 consecutive tokens aligned at
  absolute positions 128 g.  Values: per token over groups of 32 consecutive
  channels.
* Tokens not yet in a full group stay as the original bf16 K/V (the
  residual window) and are attended to unquantised.
* Decode score of a quantised token t for query q:
  s_t = n_t * (H_d q) . (code_t * s + z) * softmax_scale; of a window token:
  s_t = q . k_t * softmax_scale.  Softmax with max subtraction; output is
  sum_t p_t * v_hat_t.  softmax_scale defaults to 1 / sqrt(d).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

HEAD_DIM = 128          # d
KEY_GROUP = 128         # G: tokens per key quantisation group
VALUE_GROUP = 32        # channels per value quantisation group
MAX_CODE = 3            # INT2 levels 0..3


# ---------------------------------------------------------------------------
# Canalized Rotation (OScaR abstract; ai-papers.net "OScaRの提案手法", stage 1)
# ---------------------------------------------------------------------------

def hadamard_unnormalised(d: int = HEAD_DIM) -> np.ndarray:
    """Walsh-Hadamard matrix with entries +-1 in Sylvester (natural) order:
    Hu[i, j] = (-1)^popcount(i & j)."""
    if d <= 0 or (d & (d - 1)) != 0:
        raise ValueError("d must be a power of two")
    idx = np.arange(d)
    parity = np.zeros((d, d), dtype=np.int64)
    both = idx[:, None] & idx[None, :]
    while np.any(both):
        parity ^= both & 1
        both = both >> 1
    return np.where(parity == 1, -1.0, 1.0)


def hadamard(d: int = HEAD_DIM) -> np.ndarray:
    """Normalised Walsh-Hadamard matrix H_d = Hu / sqrt(d); symmetric and
    orthogonal."""
    return hadamard_unnormalised(d) / np.sqrt(d)


def canalized_rotation(k: np.ndarray) -> np.ndarray:
    """Rotate every key vector (last axis) by H_d: r = H_d k = (Hu k) / sqrt(d).

    Hu k is a sum of +-k_j; for bf16-valued inputs it is exact in float64, so
    every component of r carries a single rounding (the division).
    """
    d = k.shape[-1]
    return (k @ hadamard_unnormalised(d).T) / np.sqrt(d)


# ---------------------------------------------------------------------------
# Omni-Token Scaling (ai-papers.net "OScaRの提案手法", stage 2)
# ---------------------------------------------------------------------------

def omni_token_scaling(r: np.ndarray):
    """Return (n, k_hat): the L2 norm of every token and the token divided by it.

    A token whose norm is zero maps to the zero vector.
    """
    n = np.sqrt(np.sum(r * r, axis=-1))
    safe = np.where(n > 0.0, n, 1.0)
    k_hat = np.where(n[..., None] > 0.0, r / safe[..., None], 0.0)
    return n, k_hat


# ---------------------------------------------------------------------------
# Asymmetric INT2 quantiser (KIVI convention as described in the NOVA-KV
# article; OScaR abstract: INT2 per-channel paradigm)
# ---------------------------------------------------------------------------

def store_meta(x: np.ndarray, meta_bits: int = 32) -> np.ndarray:
    """Stored metadata: float32, or (meta_bits = 16) that float32 rounded to
    float16, nearest even; returned as float32 (exact either way)."""
    x32 = np.asarray(x).astype(np.float32)
    if meta_bits == 16:
        return x32.astype(np.float16).astype(np.float32)
    if meta_bits != 32:
        raise ValueError("meta_bits must be 32 or 16")
    return x32


def int2_params(x_min: np.ndarray, x_max: np.ndarray, meta_bits: int = 32):
    """Scale and zero of an asymmetric 4-level quantiser as stored: float32,
    or float16 in the 16-bit metadata layout (the float32 value rounded)."""
    s32 = ((x_max - x_min) / MAX_CODE).astype(np.float32)
    z32 = np.asarray(x_min).astype(np.float32)
    return store_meta(s32, meta_bits), store_meta(z32, meta_bits)


def int2_codes(x: np.ndarray, s32: np.ndarray, z32: np.ndarray):
    """Codes and pre-rounding values of x against broadcastable s32, z32.

    pre = (x - z) / s in float64 from the exact values of the stored
    parameters; code = clamp(round_half_even(pre), 0, 3); s == 0 gives code 0
    (and pre 0: every x of such a group equals z).
    """
    x = np.asarray(x, dtype=np.float64)
    s = np.asarray(s32, dtype=np.float64)
    z = np.asarray(z32, dtype=np.float64)
    ok = s > 0.0
    pre = np.where(ok, (x - z) / np.where(ok, s, 1.0), 0.0)
    codes = np.clip(np.rint(pre), 0, MAX_CODE).astype(np.uint8)
    return codes, pre


def int2_dequant(codes: np.ndarray, s32: np.ndarray, z32: np.ndarray) -> np.ndarray:
    return codes.astype(np.float64) * np.asarray(s32, np.float64) + np.asarray(z32, np.float64)


@dataclass
class KeyGroup:
    codes: np.ndarray   # uint8 [..., G, d]   (token, channel)
    scale: np.ndarray   # float32 [..., d]    per channel
    zero: np.ndarray    # float32 [..., d]
    norm: np.ndarray    # float32 [..., G]    per token
    pre: np.ndarray     # float64 [..., G, d] pre-rounding values


@dataclass
class ValueGroup:
    codes: np.ndarray   # uint8 [..., G, d]
    scale: np.ndarray   # float32 [..., G, d // 32]
    zero: np.ndarray    # float32 [..., G, d // 32]
    pre: np.ndarray     # float64 [..., G, d]


def quantize_key_group(k: np.ndarray, meta_bits: int = 32) -> KeyGroup:
    """OScaR key path for one group of tokens (axis -2) of bf16-valued keys.

    Steps in the pages' order: Canalized Rotation, then Omni-Token Scaling,
    then per-channel asymmetric INT2 over the group's tokens.  The codes are
    decided against the stored (possibly float16) scale and zero.
    """
    k = np.asarray(k, dtype=np.float64)
    r = canalized_rotation(k)
    n, k_hat = omni_token_scaling(r)
    s32, z32 = int2_params(k_hat.min(axis=-2), k_hat.max(axis=-2), meta_bits)
    codes, pre = int2_codes(k_hat, s32[..., None, :], z32[..., None, :])
    return KeyGroup(codes, s32, z32, store_meta(n, meta_bits), pre)


def quantize_value_group(v: np.ndarray, meta_bits: int = 32) -> ValueGroup:
    """Per-token asymmetric INT2 of values over groups of 32 channels."""
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[-1]
    vg = v.reshape(v.shape[:-1] + (d // VALUE_GROUP, VALUE_GROUP))
    s32, z32 = int2_params(vg.min(axis=-1), vg.max(axis=-1), meta_bits)
    codes, pre = int2_codes(vg, s32[..., None], z32[..., None])
    return ValueGroup(codes.reshape(v.shape), s32, z32, pre.reshape(v.shape))


def dequant_keys(g: KeyGroup) -> np.ndarray:
    """Unit-norm key estimate code * s + z (still in the rotated basis)."""
    return int2_dequant(g.codes, g.scale[..., None, :], g.zero[..., None, :])


def dequant_values(g: ValueGroup) -> np.ndarray:
    d = g.codes.shape[-1]
    c = g.codes.reshape(g.codes.shape[:-1] + (d // VALUE_GROUP, VALUE_GROUP))
    return int2_dequant(c, g.scale[..., None], g.zero[..., None]).reshape(g.codes.shape)


# ---------------------------------------------------------------------------
# Cache of one (sequence, KV head): closed groups + bf16 residual window
# ---------------------------------------------------------------------------

@dataclass
class HeadCache:
    """Quantised groups (stacked along axis 0) and the residual bf16 window."""

    keys: Optional[KeyGroup]            # arrays with leading axis = group
    values: Optional[ValueGroup]
    window_k: np.ndarray                # float64 [R, d] (bf16 values)
    window_v: np.ndarray

    @property
    def num_groups(self) -> int:
        return 0 if self.keys is None else self.keys.codes.shape[0]

    @property
    def length(self) -> int:
        return self.num_groups * KEY_GROUP + self.window_k.shape[0]


def build_head_cache(k: np.ndarray, v: np.ndarray, meta_bits: int = 32) -> HeadCache:
    """Quantise every full group of positions [128 g, 128 g + 128) of one head
    (k, v: [L, d]) and keep the remaining L mod 128 tokens as the window.
    meta_bits = 16 stores scales, zeros and norms as float16."""
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L, d = k.shape
    ng = L // KEY_GROUP
    cut = ng * KEY_GROUP
    keys = values = None
    if ng > 0:
        keys = quantize_key_group(k[:cut].reshape(ng, KEY_GROUP, d), meta_bits)
        values = quantize_value_group(v[:cut].reshape(ng, KEY_GROUP, d), meta_bits)
    return HeadCache(keys, values, k[cut:].copy(), v[cut:].copy())


# ---------------------------------------------------------------------------
# Decode attention over the packed cache
# ---------------------------------------------------------------------------

def decode_scores(q: np.ndarray, cache: HeadCache, softmax_scale: Optional[float] = None):
    """Scores of query rows q [Hg, d] against every cached token, in position
    order: quantised groups first, then the window."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    scale = (1.0 / np.sqrt(d)) if softmax_scale is None else float(softmax_scale)
    parts = []
    if cache.num_groups > 0:
        q_rot = canalized_rotation(q)                             # H_d q
        k_hat = dequant_keys(cache.keys).reshape(-1, d)           # [ng*G, d]
        n = cache.keys.norm.astype(np.float64).reshape(-1)        # [ng*G]
        parts.append((k_hat @ q_rot.T) * n[:, None] * scale)      # [T, Hg]
    if cache.window_k.shape[0] > 0:
        parts.append((cache.window_k @ q.T) * scale)
    return np.concatenate(parts, axis=0)


def decode_values(cache: HeadCache) -> np.ndarray:
    parts = []
    if cache.num_groups > 0:
        parts.append(dequant_values(cache.values).reshape(-1, cache.values.codes.shape[-1]))
    if cache.window_v.shape[0] > 0:
        parts.append(cache.window_v)
    return np.concatenate(parts, axis=0)


def softmax_attend(scores: np.ndarray, values: np.ndarray) -> np.ndarray:
    """o[h] = sum_t p[t, h] v[t] with p = softmax over t (max subtracted)."""
    m = scores.max(axis=0, keepdims=True)
    e = np.exp(scores - m)
    p = e / e.sum(axis=0, keepdims=True)
    return p.T @ values


def decode_head(q: np.ndarray, cache: HeadCache, softmax_scale: Optional[float] = None):
    """Attention output [Hg, d] of the query heads sharing one KV head."""
    if cache.length == 0:
        raise ValueError("decode over an empty cache")
    return softmax_attend(decode_scores(q, cache, softmax_scale), decode_values(cache))


def decode_attention(q: np.ndarray, caches: Sequence[Sequence[HeadCache]],
                     softmax_scale: Optional[float] = None) -> np.ndarray:
    """Batched decode: q [B, Hq, d]; caches[b][j] for KV head j.

    Query head h reads KV head h // (Hq / Hkv) (contiguous GQA grouping).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    out = np.zeros((B, Hq, d))
    for b in range(B):
        Hkv = len(caches[b])
        if Hq % Hkv != 0:
            raise ValueError("Hq must be a multiple of Hkv")
        gqa = Hq // Hkv
        for j in range(Hkv):
            out[b, j * gqa:(j + 1) * gqa] = decode_head(q[b, j * gqa:(j + 1) * gqa],
                                                      caches[b][j], softmax_scale)
    return out


def history_attention(q: np.ndarray, cache: HeadCache, softmax_scale: Optional[float] = None):
    """Chunked-prefill attention of query rows q [R, d] (the chunk's queries of
    the query heads sharing one KV head) over every token already in the
    cache: quantised groups and window, no mask (the cache precedes the
    chunk).  Returns (o [R, d], lse [R]) with lse = ln sum_t exp(s_t), so that
    the chunk's own causal part can be merged in (merge_attention)."""
    if cache.length == 0:
        raise ValueError("attention over an empty cache")
    s = decode_scores(q, cache, softmax_scale)              # [T, R]
    m = s.max(axis=0)
    e = np.exp(s - m[None, :])
    l = e.sum(axis=0)
    o = (e / l[None, :]).T @ decode_values(cache)
    return o, m + np.log(l)


def merge_attention(o1: np.ndarray, lse1: np.ndarray, o2: np.ndarray, lse2: np.ndarray):
    """Attention over the union of two disjoint key sets from the parts'
    outputs and log-sum-exps (the log-sum-exp merge of split-K decoding)."""
    mx = np.maximum(lse1, lse2)
    w1, w2 = np.exp(lse1 - mx), np.exp(lse2 - mx)
    o = (w1[:, None] * o1 + w2[:, None] * o2) / (w1 + w2)[:, None]
    return o, mx + np.log(w1 + w2)


def attention_exact(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                    softmax_scale: Optional[float] = None) -> np.ndarray:
    """Unquantised single-query attention of q [Hg, d] over k, v [L, d]."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    scale = (1.0 / np.sqrt(d)) if softmax_scale is None else float(softmax_scale)
    s = (np.asarray(k, np.float64) @ q.T) * scale
    return softmax_attend(s, np.asarray(v, np.float64))


# ---------------------------------------------------------------------------
# Variants used only for reports (not gated): order and ablations of the
# two OScaR stages (ai-papers.net "OScaRの提案手法": rotation must precede
# scaling; NOVA-KV article: KIVI = per-channel keys without either stage).
# ---------------------------------------------------------------------------

def quantize_key_group_variant(k: np.ndarray, rotate: bool, scale: bool,
                               scale_first: bool = False):
    """Return the dequantised keys (in the original basis, times the norm)
    of a variant pipeline, for error reports."""
    k = np.asarray(k, dtype=np.float64)
    x = k
    n = np.ones(k.shape[:-1])
    if scale and scale_first:
        n, x = omni_token_scaling(x)
    if rotate:
        x = canalized_rotation(x)
    if scale and not scale_first:
        n, x = omni_token_scaling(x)
    s32, z32 = int2_params(x.min(axis=-2), x.max(axis=-2))
    codes, _ = int2_codes(x, s32[..., None, :], z32[..., None, :])
    xh = int2_dequant(codes, s32[..., None, :], z32[..., None, :])
    if rotate:
        xh = xh @ hadamard(k.shape[-1])      # H_d^T = H_d: undo the rotation
    return xh * n[..., None]
