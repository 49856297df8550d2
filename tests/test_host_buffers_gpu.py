"""Decode calls with page-locked host buffers: the kernels read q and write
out in place through the device mapping.  The results must equal those of the
same calls with device buffers bit for bit; pageable host memory, and host
memory where only device memory is accepted (appended rows), must be refused
before anything is enqueued."""
import pytest
import torch

from int2_kv_cache_oscar_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


def _caches(lens, hkv, seed, n=2):
    gen = torch.Generator().manual_seed(seed)
    ks, vs = [], []
    for L in lens:
        k, v = W.make_sequence_kv(L, hkv, W.LLAMA_RECIPE, gen)
        ks.append(k)
        vs.append(v)
    out = []
    for _ in range(n):
        c = U.lib().OscarCache(len(lens), hkv, max(lens) + 256)
        U.append_all(c, list(range(len(lens))), ks, vs)
        out.append(c)
    return out


@pytest.mark.parametrize("lens", [[8192 + 77], [300, 5000, 129, 4096]])
def test_decode_host_buffers_match_device(lens):
    (c,) = _caches(lens, 8, seed=101, n=1)
    hq, B = 32, len(lens)
    q = W.make_q(B, hq, seed=102)
    ws = c.workspace(B, hq)
    o_dev = torch.empty((B, hq, 128), dtype=torch.bfloat16, device="cuda")
    c.decode(list(range(B)), q.cuda(), hq, o_dev, ws)
    q_host = q.pin_memory()
    o_host = torch.full((B, hq, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
    c.decode(list(range(B)), q_host, hq, o_host, ws)
    torch.cuda.synchronize()
    U.lib().oscar_cache_check(c.handle)
    assert torch.equal(o_host, o_dev.cpu())
    # mixed: device q, host out
    o_host2 = torch.zeros_like(o_host).pin_memory()    # zeros_like alone is pageable
    c.decode(list(range(B)), q.cuda(), hq, o_host2, ws)
    torch.cuda.synchronize()
    assert torch.equal(o_host2, o_host)


def test_append_decode_host_buffers_match_device():
    a, b = _caches([2048 + 60, 127, 1000], 2, seed=103)
    hq, B = 8, 3
    gen = torch.Generator().manual_seed(104)
    ids = [0, 1, 2]
    ws_a, ws_b = a.workspace(B, hq), b.workspace(B, hq)
    for step in range(3):        # step 0 closes the group of sequence 1 (127 -> 128 tokens)
        kn = torch.randn((B, 2, 128), generator=gen).to(torch.bfloat16)
        vn = torch.randn((B, 2, 128), generator=gen).to(torch.bfloat16)
        q = torch.randn((B, hq, 128), generator=gen).to(torch.bfloat16)
        o_dev = torch.empty((B, hq, 128), dtype=torch.bfloat16, device="cuda")
        a.append_decode(ids, kn.cuda(), vn.cuda(), q.cuda(), hq, o_dev, ws_a)
        o_host = torch.empty((B, hq, 128), dtype=torch.bfloat16).pin_memory()
        qh = q.pin_memory()                  # alive until the kernels ran
        b.append_decode(ids, kn.cuda(), vn.cuda(), qh, hq, o_host, ws_b)
        torch.cuda.synchronize()
        assert torch.equal(o_host, o_dev.cpu()), f"step {step}"
    ra, rb = U.read_arena(a), U.read_arena(b)
    for s in ids:
        assert a.length(s) == b.length(s)
        assert (U.live_bytes(a, ra, s) == U.live_bytes(b, rb, s)).all()


def test_pageable_host_buffers_are_refused():
    O_ = U.lib()
    (c,) = _caches([300], 2, seed=105, n=1)
    hq = 8
    ws = c.workspace(1, hq)
    q_dev = torch.zeros((1, hq, 128), dtype=torch.bfloat16, device="cuda")
    o_dev = torch.zeros_like(q_dev)
    q_pageable = torch.zeros((1, hq, 128), dtype=torch.bfloat16)
    o_pageable = torch.zeros_like(q_pageable)
    for q, o in [(q_pageable, o_dev), (q_dev, o_pageable)]:
        with pytest.raises(O_.OscarError) as e:
            c.decode([0], q, hq, o, ws)
        assert e.value.status == O_.OSCAR_ERR_INVALID_ARG
        assert "pageable" in str(e.value)
    kn = torch.zeros((1, 2, 128), dtype=torch.bfloat16).pin_memory()
    with pytest.raises(O_.OscarError) as e:      # the new token: device memory only
        c.append_decode([0], kn, kn.cuda(), q_dev, hq, o_dev, ws)
    assert e.value.status == O_.OSCAR_ERR_INVALID_ARG
    with pytest.raises(O_.OscarError) as e:      # appends: device memory only
        c.append([0], [0, 1], kn, kn.cuda())
    assert e.value.status == O_.OSCAR_ERR_INVALID_ARG
    assert c.length(0) == 300                    # nothing appended
    torch.cuda.synchronize()
    O_.oscar_cache_check(c.handle)


def test_prefill_host_buffers_and_refusals():
    O_ = U.lib()
    (c,) = _caches([2048 + 33], 2, seed=106, n=1)
    hq, n_q = 8, 19
    gen = torch.Generator().manual_seed(107)
    q = torch.randn((n_q, hq, 128), generator=gen).to(torch.bfloat16)
    o_dev = torch.empty((n_q, hq, 128), dtype=torch.bfloat16, device="cuda")
    l_dev = torch.empty((n_q, hq), dtype=torch.float32, device="cuda")
    O_.oscar_prefill_attention(c.handle, 0, q.cuda(), hq, 0.0, o_dev, l_dev)
    q_h = q.pin_memory()
    o_h = torch.zeros((n_q, hq, 128), dtype=torch.bfloat16).pin_memory()
    l_h = torch.zeros((n_q, hq), dtype=torch.float32).pin_memory()
    O_.oscar_prefill_attention(c.handle, 0, q_h, hq, 0.0, o_h, l_h)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_dev.cpu()) and torch.equal(l_h, l_dev.cpu())
    with pytest.raises(O_.OscarError) as e:           # pageable output
        O_.oscar_prefill_attention(c.handle, 0, q_h, hq, 0.0, torch.zeros_like(o_h), l_h)
    assert e.value.status == O_.OSCAR_ERR_INVALID_ARG


def test_bf16_reference_refuses_host_caches():
    O_ = U.lib()
    L, hkv, hq = 256, 2, 8
    kc = torch.zeros((1, hkv, L, 128), dtype=torch.bfloat16).pin_memory()
    vc = torch.zeros((1, hkv, L, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((1, hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    ws = torch.empty(O_.oscar_bf16_decode_workspace_bytes(1, hkv, hq), dtype=torch.uint8, device="cuda")
    with pytest.raises(O_.OscarError) as e:
        O_.oscar_bf16_decode_attention([0], [L], kc, vc, hkv, L, q, hq, 0.0, out, ws)
    assert e.value.status == O_.OSCAR_ERR_INVALID_ARG

