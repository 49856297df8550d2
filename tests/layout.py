"""Reader of the library's device layout, written from the description in
include/oscar.h (not from the CUDA sources): unpacks a 13,824-byte group
block into canonical arrays, and packs canonical codes into fragment order
(used only to check that the two are inverse).

Fragment words of a 128x128 matrix of 2-bit codes X[row][col]: word
F(mt, lane, j, r) holds the 16 codes with row = 16*mt + (lane >> 2) + 8*r and
col = 16*(4*j + kk) + 8*hf + 2*(lane & 3) + e, the code sitting at bits
[b, b+1], b = 16*e + 4*kk + 2*hf.  K codes store F(mt, lane, j, r) as word
(mt*32 + lane)*4 + 2*j + r ("k" order), V codes as ((mt*2 + j)*32 + lane)*2 + r
("v" order).
"""
from __future__ import annotations

import numpy as np

D = 128
G = 128
BLOCK_BYTES = 13824
OFF_KCODES, OFF_KSCALE, OFF_KZERO, OFF_KNORM, OFF_VCODES = 0, 4096, 4608, 5120, 5632
OFF_VSCALE, OFF_VZERO = 9728, 11776
# float32 value scales / zeros: token t is stored in row t ^ ((t >> 3) & 1)
VMETA_ROW = np.array([t ^ ((t >> 3) & 1) for t in range(128)])
# the same block with float16 metadata (meta_bits = 16)
BLOCK_BYTES16 = 11008
OFF16_KSCALE, OFF16_KZERO, OFF16_KNORM, OFF16_VCODES = 4096, 4352, 4608, 4864
OFF16_VSCALE, OFF16_VZERO = 8960, 9984


def block_bytes(meta_bits: int = 32) -> int:
    return BLOCK_BYTES16 if meta_bits == 16 else BLOCK_BYTES


def _word(order: str, mt: int, lane: int, j: int, r: int) -> int:
    if order == "k":
        return (mt * 32 + lane) * 4 + 2 * j + r
    if order == "v":
        return ((mt * 2 + j) * 32 + lane) * 2 + r
    raise ValueError(order)


def _index_tables(order: str):
    rows = np.zeros((1024, 16), np.int64)
    cols = np.zeros((1024, 16), np.int64)
    bits = np.zeros((1024, 16), np.int64)
    for mt in range(8):
        for lane in range(32):
            for j in range(2):
                for r in range(2):
                    w = _word(order, mt, lane, j, r)
                    n = 0
                    for kk in range(4):
                        for hf in range(2):
                            for e in range(2):
                                rows[w, n] = 16 * mt + (lane >> 2) + 8 * r
                                cols[w, n] = 16 * (4 * j + kk) + 8 * hf + 2 * (lane & 3) + e
                                bits[w, n] = 16 * e + 4 * kk + 2 * hf
                                n += 1
    return rows, cols, bits


_TABLES = {o: _index_tables(o) for o in ("k", "v")}


def unpack_fragment(words: np.ndarray, order: str = "k") -> np.ndarray:
    """uint32 [1024] (little-endian words) -> uint8 codes [128, 128] X[row][col]."""
    rows, cols, bits = _TABLES[order]
    words = np.asarray(words, dtype=np.uint32).reshape(1024)
    vals = (words[:, None].astype(np.int64) >> bits) & 3
    out = np.zeros((G, D), np.uint8)
    out[rows, cols] = vals
    return out


def pack_fragment(codes: np.ndarray, order: str = "k") -> np.ndarray:
    rows, cols, bits = _TABLES[order]
    codes = np.asarray(codes, np.int64)
    vals = codes[rows, cols] << bits
    return np.bitwise_or.reduce(vals, axis=1).astype(np.uint32)


def parse_block(raw: np.ndarray, meta_bits: int = 32) -> dict:
    """raw: uint8 [13824] (or [11008] with float16 metadata) -> canonical
    arrays of one (group, kv head); metadata returned as float32."""
    if meta_bits == 16:
        raw = np.ascontiguousarray(np.asarray(raw, np.uint8).reshape(BLOCK_BYTES16))
        kcodes = unpack_fragment(raw[OFF_KCODES:OFF_KCODES + 4096].view("<u4"))
        f16 = lambda a, n: raw[a:a + 2 * n].view("<f2").astype(np.float32)
        vcodes_t = unpack_fragment(raw[OFF16_VCODES:OFF16_VCODES + 4096].view("<u4"), "v")
        return dict(kcodes=kcodes, kscale=f16(OFF16_KSCALE, 128), kzero=f16(OFF16_KZERO, 128),
                    knorm=f16(OFF16_KNORM, 128), vcodes=vcodes_t.T.copy(),
                    vscale=f16(OFF16_VSCALE, 512).reshape(G, 4), vzero=f16(OFF16_VZERO, 512).reshape(G, 4))
    raw = np.ascontiguousarray(np.asarray(raw, np.uint8).reshape(BLOCK_BYTES))
    kcodes = unpack_fragment(raw[OFF_KCODES:OFF_KCODES + 4096].view("<u4"))        # [token, ch]
    kscale = raw[OFF_KSCALE:OFF_KSCALE + 512].view("<f4").copy()
    kzero = raw[OFF_KZERO:OFF_KZERO + 512].view("<f4").copy()
    knorm = raw[OFF_KNORM:OFF_KNORM + 512].view("<f4").copy()
    vcodes_t = unpack_fragment(raw[OFF_VCODES:OFF_VCODES + 4096].view("<u4"), "v")  # [ch, token]
    rows = VMETA_ROW                                                               # token t in row rows[t]
    vscale = raw[OFF_VSCALE:OFF_VSCALE + 2048].view("<f4").reshape(G, 4)[rows].copy()
    vzero = raw[OFF_VZERO:OFF_VZERO + 2048].view("<f4").reshape(G, 4)[rows].copy()
    return dict(kcodes=kcodes, kscale=kscale, kzero=kzero, knorm=knorm,
                vcodes=vcodes_t.T.copy(), vscale=vscale, vzero=vzero)


def bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    u = np.asarray(u16, np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def parse_window(raw: np.ndarray, n: int):
    """raw: uint8 [65536] window of one (slot, head) -> (k [n, d], v [n, d]) float64."""
    raw = np.ascontiguousarray(np.asarray(raw, np.uint8).reshape(65536))
    k = bf16_bits_to_f64(raw[:32768].view("<u2").reshape(G, D)[:n])
    v = bf16_bits_to_f64(raw[32768:].view("<u2").reshape(G, D)[:n])
    return k, v
