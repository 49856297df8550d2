"""Decode with float32 outputs (oscar_decode_attention_f32) against the
oracle's float64 attention over the GPU's own cache, at a plain 2e-3 max-abs
(no bf16 output rounding to absorb kernel error), and the bf16 decode as that
float32 output rounded to nearest even.  The worst absolute and relative
errors are printed (relative to max(|ref|, 1e-2))."""
import numpy as np
import pytest
import torch

from int2_kv_cache_oscar_gb300 import workloads as W
from oracle import oscar_oracle as O
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu

F32_ABS = 2e-3


def _bf16_round(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).float().double().numpy()


def _run(lens, hkv, hq, seed, meta_bits=32, scale=0.0):
    gen = torch.Generator().manual_seed(seed)
    ks, vs = [], []
    for L in lens:
        k, v = W.make_sequence_kv(L, hkv, W.LLAMA_RECIPE, gen)
        ks.append(k)
        vs.append(v)
    cache = U.lib().OscarCache(len(lens), hkv, max(lens) + 128, meta_bits=meta_bits)
    U.append_all(cache, list(range(len(lens))), ks, vs, chunk=2048)
    q = W.make_q(len(lens), hq, seed=seed + 1).cuda()
    ids = list(range(len(lens)))
    ws = cache.workspace(len(lens), hq)
    o32 = torch.empty((len(lens), hq, 128), dtype=torch.float32, device="cuda")
    o16 = torch.empty((len(lens), hq, 128), dtype=torch.bfloat16, device="cuda")
    cache.decode_f32(ids, q, hq, o32, ws, softmax_scale=scale)
    cache.decode(ids, q, hq, o16, ws, softmax_scale=scale)
    U.lib().oscar_cache_check(cache.handle)
    arena = U.read_arena(cache)
    g32, g16, qn = U.f64(o32), U.f64(o16), U.f64(q)
    assert np.array_equal(g16, _bf16_round(g32)), "bf16 output is not the float32 output rounded"
    gq = hq // hkv
    worst_abs = worst_rel = 0.0
    for i in range(len(lens)):
        for j in range(hkv):
            ref = O.decode_head(qn[i, gq * j:gq * (j + 1)], U.gpu_head(cache, arena, i, j),
                                None if scale == 0.0 else scale)
            d = np.abs(g32[i, gq * j:gq * (j + 1)] - ref)
            assert np.all(np.isfinite(g32[i, gq * j:gq * (j + 1)]))
            worst_abs = max(worst_abs, float(d.max()))
            worst_rel = max(worst_rel, float((d / np.maximum(np.abs(ref), 1e-2)).max()))
            assert d.max() <= F32_ABS, f"seq {i} head {j}: max |f32 - oracle| {d.max():.3e} > {F32_ABS}"
    print(f"f32 decode {lens} hq {hq} meta {meta_bits}: max abs {worst_abs:.2e}, max rel {worst_rel:.2e}")
    cache.close()
    return worst_abs


@pytest.mark.parametrize("lens,hkv,hq", [([8192 + 37], 8, 32), ([1, 100, 128, 300, 5000], 8, 32),
                                          ([1024], 1, 4), ([3000, 700], 2, 16)])
def test_f32_output_gate(lens, hkv, hq):
    _run(lens, hkv, hq, seed=31)


def test_f32_output_gate_meta16_and_scale():
    _run([4096 + 90, 513], 8, 32, seed=37, meta_bits=16, scale=0.3)


def test_f32_host_output_buffer():
    """The float32 output may be page-locked host memory, like the bf16 one."""
    gen = torch.Generator().manual_seed(41)
    k, v = W.make_sequence_kv(2000, 8, W.LLAMA_RECIPE, gen)
    cache = U.lib().OscarCache(1, 8, 2048)
    U.append_all(cache, [0], [k], [v])
    q = W.make_q(1, 32, seed=42).cuda()
    ws = cache.workspace(1, 32)
    dev = torch.empty((1, 32, 128), dtype=torch.float32, device="cuda")
    host = torch.empty((1, 32, 128), dtype=torch.float32).pin_memory()
    cache.decode_f32([0], q, 32, dev, ws)
    cache.decode_f32([0], q, 32, host, ws)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), host)
    with pytest.raises(ValueError):            # the binding checks the output dtype
        cache.decode_f32([0], q, 32, torch.empty((1, 32, 128), dtype=torch.bfloat16, device="cuda"), ws)
