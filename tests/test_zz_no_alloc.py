"""The decode entry point that allocates nothing (oscar_decode_attention_noalloc).

It serves callers that cannot allocate device memory where they decode, by
keeping the split-K partials in a fixed device array inside the library.
Here it is called through the C ABI and must give the same outputs as the
regular oscar_decode_attention (within the decode tolerance), on two calls in
a row: the shared array keeps the previous call's contents, which must not
leak into the next call.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from int2_kv_cache_oscar_gb300 import workloads as W
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_workspace_decode_twice():
    O_ = U.lib()
    lens = [3000, 129, 8192 + 17]
    gen = torch.Generator().manual_seed(91)
    ks, vs = [], []
    for L in lens:
        k, v = W.make_sequence_kv(L, 8, W.LLAMA_RECIPE, gen)
        ks.append(k)
        vs.append(v)
    cache = O_.OscarCache(3, 8, 8192 + 128)
    U.append_all(cache, [2, 0, 1], ks, vs, chunk=1500)
    slots = [2, 0, 1]
    for call in range(2):
        q = W.make_q(3, 32, seed=92 + call).cuda()
        ref = torch.empty((3, 32, 128), dtype=torch.bfloat16, device="cuda")
        cache.decode(slots, q, 32, ref, cache.workspace(3, 32))
        got = torch.full((3, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        O_.oscar_decode_attention_noalloc(cache.handle, slots, q, 32, 0.0, got)
        O_.oscar_cache_check(cache.handle)
        g, r = U.f64(got), U.f64(ref)
        assert np.all(np.isfinite(g))
        P.assert_decode(g, r, f"no-alloc call {call}")
    # a call needing more partials than the built-in scratch is refused before
    # anything runs: 256 sequences x 8 KV heads of records (buffers sized for
    # the call all the same)
    n_big = 256
    big = O_.OscarCache(n_big, 8, 128)
    q_big = torch.zeros((n_big, 32, 128), dtype=torch.bfloat16, device="cuda")
    o_big = torch.empty_like(q_big)
    with pytest.raises(O_.OscarError) as e:
        O_.oscar_decode_attention_noalloc(big.handle, list(range(n_big)), q_big, 32, 0.0, o_big)
    assert e.value.status == O_.OSCAR_ERR_CAPACITY
