"""Helpers of the GPU parity tests: build caches through the C ABI, read the
arena back and turn it into the oracle's canonical form."""
from __future__ import annotations

import numpy as np
import torch

from oracle import oscar_oracle as O
from tests import layout


def lib():
    from int2_kv_cache_oscar_gb300 import oscar   # raises if liboscar.so is missing
    return oscar


def f64(t: torch.Tensor) -> np.ndarray:
    """bf16/fp32 tensor -> float64 numpy (exact for bf16)."""
    return t.detach().float().cpu().double().numpy()


def append_all(cache, slots, ks, vs, chunk=None, device="cuda"):
    """Append sequences ks[i], vs[i] ([L_i, Hkv, d] bf16) to slots[i], all in
    the same calls, `chunk` tokens per sequence per call (None = at once)."""
    pos = [0] * len(slots)
    while True:
        ids, pieces_k, pieces_v, cu = [], [], [], [0]
        for i, s in enumerate(slots):
            L = ks[i].shape[0]
            if pos[i] >= L:
                continue
            n = L - pos[i] if chunk is None else min(chunk if isinstance(chunk, int) else chunk(i, pos[i]),
                                                    L - pos[i])
            ids.append(s)
            pieces_k.append(ks[i][pos[i]:pos[i] + n])
            pieces_v.append(vs[i][pos[i]:pos[i] + n])
            cu.append(cu[-1] + n)
            pos[i] += n
        if not ids:
            break
        k = torch.cat(pieces_k).to(device).contiguous()
        v = torch.cat(pieces_v).to(device).contiguous()
        cache.append(ids, cu, k, v)


def read_arena(cache) -> np.ndarray:
    torch.cuda.synchronize()
    return cache.arena.cpu().numpy()


def gpu_head(cache, arena: np.ndarray, slot: int, head: int) -> O.HeadCache:
    """The cache of (slot, head) as stored on the GPU, in the oracle's form."""
    O_ = lib()
    L = cache.length(slot)
    ng, w = L // 128, L % 128
    keys = values = None
    if ng > 0:
        parts = []
        for g in range(ng):
            off = O_.oscar_cache_block_offset(cache.handle, slot, head, g)
            mb = getattr(cache, "meta_bits", 32)
            parts.append(layout.parse_block(arena[off:off + layout.block_bytes(mb)], mb))
        st = {k: np.stack([p[k] for p in parts]) for k in parts[0]}
        keys = O.KeyGroup(st["kcodes"], st["kscale"], st["kzero"], st["knorm"], None)
        values = O.ValueGroup(st["vcodes"], st["vscale"], st["vzero"], None)
    off = O_.oscar_cache_window_offset(cache.handle, slot, head)
    wk, wv = layout.parse_window(arena[off:off + 65536], w)
    return O.HeadCache(keys, values, wk, wv)


def oracle_head(k: torch.Tensor, v: torch.Tensor, head: int, meta_bits: int = 32) -> O.HeadCache:
    return O.build_head_cache(f64(k[:, head]), f64(v[:, head]), meta_bits)


def live_bytes(cache, arena: np.ndarray, slot: int) -> np.ndarray:
    """Concatenated bytes that hold state for `slot`: its value-scale and
    |value zero| maxima, every closed group block and the occupied window rows
    of every head."""
    O_ = lib()
    L = cache.length(slot)
    ng, w = L // 128, L % 128
    hkv = cache.num_kv_heads
    zoff = 256 + cache.cfg.max_batch * hkv * 4
    parts = [arena[256 + slot * hkv * 4: 256 + (slot + 1) * hkv * 4],
             arena[zoff + slot * hkv * 4: zoff + (slot + 1) * hkv * 4]]
    for h in range(hkv):
        for g in range(ng):
            off = O_.oscar_cache_block_offset(cache.handle, slot, h, g)
            parts.append(arena[off:off + layout.block_bytes(getattr(cache, "meta_bits", 32))])
        off = O_.oscar_cache_window_offset(cache.handle, slot, h)
        parts.append(arena[off:off + w * 256])
        parts.append(arena[off + 32768:off + 32768 + w * 256])
    return np.concatenate(parts)
