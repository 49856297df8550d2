"""Failure detection without a GPU fault: a bounded device wait that runs out.

The test hook arms the next INT2 decode so that one bulk copy of its first CTA
is never issued and its waits give up after 2^14 polls.  The kernel must
return (no hang), flag the arena, and oscar_cache_check must report
OSCAR_ERR_DEVICE_TIMEOUT; the context stays usable and the next decode is
correct (checked against the oracle over the GPU's cache)."""
import numpy as np
import pytest
import torch

from int2_kv_cache_oscar_gb300 import workloads as W
from oracle import oscar_oracle as O
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_the_cache_recovers():
    O_ = U.lib()
    gen = torch.Generator().manual_seed(61)
    k, v = W.make_sequence_kv(4096 + 50, 8, W.LLAMA_RECIPE, gen)
    cache = O_.OscarCache(1, 8, 8192)
    U.append_all(cache, [0], [k], [v])
    q = W.make_q(1, 32, seed=62).cuda()
    out = torch.empty((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    ws = cache.workspace(1, 32)
    O_.oscar_cache_check(cache.handle)                      # clean before

    O_.oscar_test_arm_wait_timeout()
    cache.decode([0], q, 32, out, ws)
    with pytest.raises(O_.OscarError) as e:
        O_.oscar_cache_check(cache.handle)                  # synchronises: the kernel returned
    assert e.value.status == O_.OSCAR_ERR_DEVICE_TIMEOUT
    O_.oscar_cache_check(cache.handle)                      # the check cleared the flag

    # the next decode on the same cache is unaffected
    cache.decode([0], q, 32, out, ws)
    O_.oscar_cache_check(cache.handle)
    arena = U.read_arena(cache)
    got, qn = U.f64(out), U.f64(q)
    for j in range(8):
        ref = O.decode_head(qn[0, 4 * j:4 * j + 4], U.gpu_head(cache, arena, 0, j))
        P.assert_decode(got[0, 4 * j:4 * j + 4], ref, f"head {j} after the timeout")
    cache.close()
