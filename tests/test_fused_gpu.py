"""GPU tests of oscar_append_decode (one decode step: append a token to each
sequence, then attend).

It must give exactly what oscar_quantize_append (one row per sequence)
followed by oscar_decode_attention gives, on steps that only extend the
window (one launch) and on steps that close a group (quantiser first), and
leave the same cache behind; its output is also checked against the oracle
over the GPU's cache, like every decode.
"""
import numpy as np
import pytest
import torch

from int2_kv_cache_oscar_gb300 import workloads as W
from oracle import oscar_oracle as O
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu

HKV, HQ = 2, 8


def _prefilled(lens, seed):
    ks, vs = [], []
    gen = torch.Generator().manual_seed(seed)
    for L in lens:
        k, v = W.make_sequence_kv(L, HKV, W.LLAMA_RECIPE, gen)
        ks.append(k)
        vs.append(v)
    caches = []
    for _ in range(2):
        c = U.lib().OscarCache(len(lens), HKV, 1024)
        U.append_all(c, list(range(len(lens))), ks, vs)
        caches.append(c)
    return caches


def test_append_decode_matches_separate_calls():
    lens = [125, 300, 1, 255]     # step 0 closes a group of sequence 3, step 2 one of sequence 0
    ids = list(range(len(lens)))
    a, b = _prefilled(lens, seed=31)
    gen = torch.Generator().manual_seed(32)
    wa, wb = a.workspace(len(ids), HQ), b.workspace(len(ids), HQ)
    oa = torch.empty((len(ids), HQ, 128), dtype=torch.bfloat16, device="cuda")
    ob = torch.empty_like(oa)
    for step in range(6):
        kn = torch.randn((len(ids), HKV, 128), generator=gen).to(torch.bfloat16).cuda()
        vn = torch.randn((len(ids), HKV, 128), generator=gen).to(torch.bfloat16).cuda()
        q = torch.randn((len(ids), HQ, 128), generator=gen).to(torch.bfloat16).cuda()
        a.append(ids, list(range(len(ids) + 1)), kn, vn)
        a.decode(ids, q, HQ, oa, wa)
        b.append_decode(ids, kn, vn, q, HQ, ob, wb)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), f"step {step}: fused output differs"
        for i, s in enumerate(ids):
            assert a.length(s) == b.length(s) == lens[i] + step + 1
        if step in (0, 1, 2, 5):
            arena = U.read_arena(b)
            got, qn = U.f64(ob), U.f64(q)
            for i, s in enumerate(ids):
                for j in range(HKV):
                    ref = O.decode_head(qn[i, j * 4:(j + 1) * 4], U.gpu_head(b, arena, s, j))
                    P.assert_decode(got[i, j * 4:(j + 1) * 4], ref, f"step {step} seq {s} head {j}")
    ra, rb = U.read_arena(a), U.read_arena(b)
    for s in ids:
        assert np.array_equal(U.live_bytes(a, ra, s), U.live_bytes(b, rb, s))
    U.lib().oscar_cache_check(b.handle)


def test_append_decode_bad_args_change_nothing():
    O_ = U.lib()
    (c, _) = _prefilled([10, 20], seed=33)
    kn = torch.zeros((2, HKV, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((2, HQ, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((2, HQ, 128), dtype=torch.bfloat16, device="cuda")
    ws = c.workspace(2, HQ)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(TypeError):                          # the binding refuses a missing buffer
        O_.oscar_append_decode(c.handle, [0, 1], None, kn, q, HQ, 0.0, out, ws)
    with pytest.raises(O_.OscarError) as e:
        O_.oscar_append_decode(c.handle, [0, 1], kn, kn, q, HQ, 0.0, out, small)
    assert e.value.status == O_.OSCAR_ERR_CAPACITY
    with pytest.raises(O_.OscarError) as e:
        O_.oscar_append_decode(c.handle, [0, 0], kn, kn, q, HQ, 0.0, out, ws)
    assert e.value.status == O_.OSCAR_ERR_INVALID_ARG
    assert c.length(0) == 10 and c.length(1) == 20


def test_append_decode_gqa8_matches_separate_calls():
    """8 query heads per KV head: the fused step runs two decode passes, each
    storing the new token; outputs and cache bytes equal the separate calls'."""
    lens = [127, 300]             # step 0 closes a group of sequence 0
    ids = list(range(len(lens)))
    hq = 8 * HKV
    a, b = _prefilled(lens, seed=33)
    gen = torch.Generator().manual_seed(34)
    wa, wb = a.workspace(len(ids), hq), b.workspace(len(ids), hq)
    oa = torch.empty((len(ids), hq, 128), dtype=torch.bfloat16, device="cuda")
    ob = torch.empty_like(oa)
    for step in range(3):
        kn = torch.randn((len(ids), HKV, 128), generator=gen).to(torch.bfloat16).cuda()
        vn = torch.randn((len(ids), HKV, 128), generator=gen).to(torch.bfloat16).cuda()
        q = torch.randn((len(ids), hq, 128), generator=gen).to(torch.bfloat16).cuda()
        a.append(ids, list(range(len(ids) + 1)), kn, vn)
        a.decode(ids, q, hq, oa, wa)
        b.append_decode(ids, kn, vn, q, hq, ob, wb)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), f"step {step}: fused output differs"
        arena = U.read_arena(b)
        got, qn = U.f64(ob), U.f64(q)
        for i, s in enumerate(ids):
            for j in range(HKV):
                ref = O.decode_head(qn[i, j * 8:(j + 1) * 8], U.gpu_head(b, arena, s, j))
                P.assert_decode(got[i, j * 8:(j + 1) * 8], ref, f"gqa 8 step {step} seq {s} head {j}")
    ra, rb = U.read_arena(a), U.read_arena(b)
    for s in ids:
        assert np.array_equal(U.live_bytes(a, ra, s), U.live_bytes(b, rb, s))
