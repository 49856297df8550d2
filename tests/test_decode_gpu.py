"""GPU parity of oscar_decode_attention (INT2 split-K + combine) and of the
BF16 reference decode.

Gate: the CUDA output against the oracle's float64 attention over the SAME
cache read back from the GPU (so that quantisation boundary differences do
not enter), |o_gpu - o_ref| <= 2e-3 + half a bf16 ulp of o_ref.  The error
against the oracle's own cache and against unquantised attention is printed.
"""
import math

import numpy as np
import pytest
import torch

from int2_kv_cache_oscar_gb300 import workloads as W
from oracle import oscar_oracle as O
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu


def _decode(cache, slots, q, hq, scale=0.0):
    O_ = U.lib()
    out = torch.empty((len(slots), hq, 128), dtype=torch.bfloat16, device="cuda")
    ws = cache.workspace(len(slots), hq)
    cache.decode(slots, q.cuda().contiguous(), hq, out, ws, softmax_scale=scale)
    O_.oscar_cache_check(cache.handle)
    return U.f64(out)


def _check(cache, slots, ks, vs, q, hq, scale=None, what=""):
    """Decode on the GPU and compare with the oracle over the GPU's cache."""
    got = _decode(cache, slots, q, hq, 0.0 if scale is None else scale)
    arena = U.read_arena(cache)
    hkv = cache.num_kv_heads
    gqa = hq // hkv
    qn = U.f64(q)
    worst = worst_own = worst_exact = worst_ulp = 0.0
    for i, s in enumerate(slots):
        for j in range(hkv):
            ref = O.decode_head(qn[i, j * gqa:(j + 1) * gqa], U.gpu_head(cache, arena, s, j), scale)
            worst = max(worst, P.assert_decode(got[i, j * gqa:(j + 1) * gqa], ref, f"{what} seq {s} head {j}"))
            worst_ulp = max(worst_ulp, P.bf16_ulp_err(got[i, j * gqa:(j + 1) * gqa], ref))
            if ks is not None:
                own = O.decode_head(qn[i, j * gqa:(j + 1) * gqa], U.oracle_head(ks[i], vs[i], j), scale)
                worst_own = max(worst_own, float(np.abs(got[i, j * gqa:(j + 1) * gqa] - own).max()))
                ex = O.attention_exact(qn[i, j * gqa:(j + 1) * gqa], U.f64(ks[i][:, j]), U.f64(vs[i][:, j]), scale)
                worst_exact = max(worst_exact, float(np.abs(got[i, j * gqa:(j + 1) * gqa] - ex).max()))
    print(f"{what}: max|gpu-oracle(gpu cache)|={worst:.2e} ({worst_ulp:.3f} bf16 ulp)  "
          f"vs oracle cache={worst_own:.2e}  vs unquantised={worst_exact:.2e}")
    return got


def test_tiny_layer_decode():
    w = W.tiny_layer()
    ks, vs, q = W.make_workload_tensors(w)
    cache = U.lib().OscarCache(1, 1, 1024)
    U.append_all(cache, [0], ks, vs)
    _check(cache, [0], ks, vs, q, 4, what="tiny")


@pytest.mark.parametrize("L", [8192, 8192 + 100, 100, 1, 128, 129])
def test_llama_layer_decode(L):
    w = W.llama_layer(L)
    ks, vs, q = W.make_workload_tensors(w)
    cache = U.lib().OscarCache(1, 8, max(L, 128))
    U.append_all(cache, [0], ks, vs)
    _check(cache, [0], ks, vs, q, 32, what=f"llama L={L}")


def test_ragged_batch_decode_and_split_invariance():
    lens = [1, 100, 128, 129, 3000, 5000, 255, 7]
    gen = torch.Generator().manual_seed(21)
    ks, vs = [], []
    for L in lens:
        k, v = W.make_sequence_kv(L, 8, W.LLAMA_RECIPE, gen)
        ks.append(k)
        vs.append(v)
    q = W.make_q(len(lens), 32, seed=22)
    slots = [7, 3, 0, 5, 1, 6, 2, 4]
    cache = U.lib().OscarCache(8, 8, 5120)
    U.append_all(cache, slots, ks, vs, chunk=700)
    got = _check(cache, slots, ks, vs, q, 32, what="ragged batch")
    # each sequence alone (different split-K partition) gives the same answer
    for i in [4, 5, 3]:
        alone = _decode(cache, [slots[i]], q[i:i + 1], 32)
        assert np.abs(alone[0] - got[i]).max() <= 2 * 2.0 ** -8 * max(1.0, np.abs(got[i]).max())


@pytest.mark.parametrize("gqa", [1, 2, 3, 4, 5, 6, 7, 8, 12, 16])
def test_gqa_group_sizes(gqa):
    """One pass serves up to 8 query heads per KV head (5 to 8 as two head
    sets reading each block once, the second one partial below 8); larger
    ratios run as several passes (12 = 8 + 4, 16 = 8 + 8)."""
    hkv = 4
    hq = hkv * gqa
    gen = torch.Generator().manual_seed(30 + gqa)
    k, v = W.make_sequence_kv(1000, hkv, W.LLAMA_RECIPE, gen)
    q = W.make_q(1, hq, seed=40 + gqa)
    cache = U.lib().OscarCache(1, hkv, 1024)
    U.append_all(cache, [0], [k], [v])
    _check(cache, [0], [k], [v], q, hq, what=f"gqa={gqa}")


def test_softmax_scale_and_zero_query():
    gen = torch.Generator().manual_seed(50)
    k, v = W.make_sequence_kv(600, 8, W.LLAMA_RECIPE, gen)
    q = W.make_q(1, 32, seed=51)
    cache = U.lib().OscarCache(1, 8, 1024)
    U.append_all(cache, [0], [k], [v])
    _check(cache, [0], [k], [v], q, 32, scale=0.3, what="scale 0.3")
    _check(cache, [0], [k], [v], torch.zeros_like(q), 32, what="q = 0")


def test_append_decode_stream():
    """Decode after every single-token append: groups close mid-stream and the
    window rolls over (the serving pattern)."""
    gen = torch.Generator().manual_seed(60)
    k, v = W.make_sequence_kv(400, 8, W.LLAMA_RECIPE, gen)
    q = W.make_q(1, 32, seed=61)
    O_ = U.lib()
    cache = O_.OscarCache(1, 8, 512)
    U.append_all(cache, [0], [k[:250]], [v[:250]])
    for L in range(250, 400):
        cache.append([0], [0, 1], k[L:L + 1].cuda(), v[L:L + 1].cuda())
        if L % 37 == 0 or L in (255, 256, 383, 384):
            _check(cache, [0], [k[:L + 1]], [v[:L + 1]], q, 32, what=f"stream L={L + 1}")


def test_decode_bad_args():
    O_ = U.lib()
    cache = O_.OscarCache(2, 8, 256)
    q = W.make_q(1, 32, seed=1).cuda()
    out = torch.empty((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    ws = cache.workspace(1, 32)
    with pytest.raises(O_.OscarError):
        cache.decode([0], q, 32, out, ws)                  # empty sequence
    gen = torch.Generator().manual_seed(2)
    k, v = W.make_sequence_kv(200, 8, W.LLAMA_RECIPE, gen)
    U.append_all(cache, [0], [k], [v])
    q36 = torch.zeros((1, 36, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(O_.OscarError) as e:
        cache.decode([0], q36, 36, torch.empty_like(q36), ws)   # 36 % 8 != 0
    assert e.value.status == O_.OSCAR_ERR_INVALID_ARG
    with pytest.raises(O_.OscarError) as e:
        cache.decode([0], q, 32, out, ws[:64])             # workspace too small
    assert e.value.status == O_.OSCAR_ERR_CAPACITY


# ------------------------------------------------------------ bf16 reference

def _bf16_cache(ks, vs, max_len):
    B = len(ks)
    hkv = ks[0].shape[1]
    kc = torch.zeros((B, hkv, max_len, 128), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    for b in range(B):
        L = ks[b].shape[0]
        kc[b, :, :L] = ks[b].transpose(0, 1)
        vc[b, :, :L] = vs[b].transpose(0, 1)
    return kc.cuda(), vc.cuda()


@pytest.mark.parametrize("lens", [[8192], [1, 63, 64, 65, 1000, 2047]])
def test_bf16_reference_decode(lens):
    O_ = U.lib()
    gen = torch.Generator().manual_seed(70)
    ks, vs = [], []
    for L in lens:
        k, v = W.make_sequence_kv(L, 8, W.LLAMA_RECIPE, gen)
        ks.append(k)
        vs.append(v)
    max_len = max(lens)
    kc, vc = _bf16_cache(ks, vs, max_len)
    q = W.make_q(len(lens), 32, seed=71)
    out = torch.empty((len(lens), 32, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(O_.oscar_bf16_decode_workspace_bytes(len(lens), 8, 32), dtype=torch.uint8,
                     device="cuda")
    O_.oscar_bf16_decode_attention(list(range(len(lens))), lens, kc, vc, 8, max_len, q.cuda(), 32, 0.0,
                                   out, ws)
    torch.cuda.synchronize()
    got = U.f64(out)
    qn = U.f64(q)
    worst = 0.0
    for b in range(len(lens)):
        for j in range(8):
            ref = O.attention_exact(qn[b, 4 * j:4 * j + 4], U.f64(ks[b][:, j]), U.f64(vs[b][:, j]))
            worst = max(worst, P.assert_decode(got[b, 4 * j:4 * j + 4], ref, f"bf16 ref seq {b} head {j}"))
    print("bf16 reference max err", worst)


def test_bf16_reference_decode_gqa8():
    """The BF16 reference with 8 query heads per KV head (two passes)."""
    O_ = U.lib()
    gen = torch.Generator().manual_seed(72)
    L, hkv, hq = 3000, 2, 16
    k, v = W.make_sequence_kv(L, hkv, W.LLAMA_RECIPE, gen)
    kc, vc = _bf16_cache([k], [v], L)
    q = W.make_q(1, hq, seed=73)
    out = torch.empty((1, hq, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(O_.oscar_bf16_decode_workspace_bytes(1, hkv, hq), dtype=torch.uint8, device="cuda")
    O_.oscar_bf16_decode_attention([0], [L], kc, vc, hkv, L, q.cuda(), hq, 0.0, out, ws)
    torch.cuda.synchronize()
    got, qn = U.f64(out), U.f64(q)
    for j in range(hkv):
        ref = O.attention_exact(qn[0, 8 * j:8 * j + 8], U.f64(k[:, j]), U.f64(v[:, j]))
        P.assert_decode(got[0, 8 * j:8 * j + 8], ref, f"bf16 ref gqa 8 head {j}")



def test_decode_captured_in_cuda_graph():
    """A decode call enqueues only kernel launches (no synchronisation, no
    allocation), so it can be captured in a CUDA graph; the plan (lengths,
    unit split) is fixed at capture.  Replays of the graph with new query
    values in the same buffer must equal eager calls bit for bit."""
    lens = [3000, 129, 8192 + 50]
    gen = torch.Generator().manual_seed(31)
    ks, vs = [], []
    for L in lens:
        k, v = W.make_sequence_kv(L, 8, W.LLAMA_RECIPE, gen)
        ks.append(k)
        vs.append(v)
    cache = U.lib().OscarCache(3, 8, max(lens))
    U.append_all(cache, [0, 1, 2], ks, vs, chunk=1000)
    hq, B = 32, len(lens)
    q = torch.empty((B, hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    ws = cache.workspace(B, hq)
    q.copy_(W.make_q(B, hq, seed=32))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        cache.decode([0, 1, 2], q, hq, out, ws)          # warm the launch path outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cache.decode([0, 1, 2], q, hq, out, ws)
    for seed in (33, 34):
        q.copy_(W.make_q(B, hq, seed=seed))
        g.replay()
        torch.cuda.synchronize()
        replayed = out.clone()
        eager = torch.empty_like(out)
        cache.decode([0, 1, 2], q, hq, eager, cache.workspace(B, hq))
        torch.cuda.synchronize()
        assert torch.equal(replayed, eager), f"seed {seed}"
    U.lib().oscar_cache_check(cache.handle)


def test_sixteen_kv_heads():
    """16 KV heads (GQA 4, 64 query heads): quantise and decode across the
    wider head dimension of every launch, two ragged sequences."""
    lens = [2 * 128 + 33, 5 * 128]
    gen = torch.Generator().manual_seed(41)
    ks, vs = [], []
    for L in lens:
        k, v = W.make_sequence_kv(L, 16, W.LLAMA_RECIPE, gen)
        ks.append(k)
        vs.append(v)
    cache = U.lib().OscarCache(2, 16, 1024)
    U.append_all(cache, [0, 1], ks, vs, chunk=200)
    q = W.make_q(2, 64, seed=42)
    _check(cache, [0, 1], ks, vs, q, 64, what="16 KV heads")
