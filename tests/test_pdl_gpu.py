"""Decode launched as a programmatic dependent of the kernel before it.

The main kernel copies blocks of settled groups (closed before the previous
decode call on the same stream) before its grid dependency wait.  These tests
check the host's record of which groups are settled, step by step through
appends, decodes, resets and a change of stream, and that outputs do not
depend on it: back-to-back decodes, a decode on a fresh stream, a decode right
after an append that closes groups, and a decode whose query is written by the
kernel just before it all match the oracle over the GPU's cache."""
import pytest
import torch

from int2_kv_cache_oscar_gb300 import workloads as W
from oracle import oscar_oracle as O
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu

ALL = 2 ** 31 - 1


def _kv(n, seed):
    gen = torch.Generator().manual_seed(seed)
    k, v = W.make_sequence_kv(n, 8, W.LLAMA_RECIPE, gen)
    return k.cuda(), v.cuda()


def _check_out(cache, out, q, slots):
    O_ = U.lib()
    O_.oscar_cache_check(cache.handle)
    arena = U.read_arena(cache)
    got, qn = U.f64(out), U.f64(q)
    for i, s in enumerate(slots):
        for j in range(8):
            ref = O.decode_head(qn[i, 4 * j:4 * j + 4], U.gpu_head(cache, arena, s, j))
            P.assert_decode(got[i, 4 * j:4 * j + 4], ref, f"slot {s} head {j}")


def test_settled_groups_follow_appends_decodes_and_streams():
    O_ = U.lib()
    cache = O_.OscarCache(3, 8, 4096)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    k, v = _kv(1408, 71)
    q = W.make_q(2, 32, seed=72).cuda()
    out = torch.empty((2, 32, 128), dtype=torch.bfloat16, device="cuda")
    ws = cache.workspace(3, 32)
    st = O_.oscar_test_settled_groups
    torch.cuda.synchronize()                              # inputs were made on the default stream
    with torch.cuda.stream(s1):
        cache.append([0, 1], [0, 1000, 1300], k[:1300], v[:1300])   # slot 0: groups 0-6, slot 1: 0-1
        assert st(cache, [0, 1, 2], s1) == [0, 0, 0]                  # no decode yet
        cache.decode([0, 1], q, 32, out, ws)
        assert st(cache, [0, 1, 2], s1) == [ALL, ALL, 0]              # slot 2 was not decoded
        assert st(cache, [0, 1], s2) == [0, 0]                        # another stream: nothing
        cache.append([0], [0, 300], k[1000:1300], v[1000:1300])       # 1000 -> 1300 closes groups 7-9
        cache.append([1], [0, 10], k[1300:1310], v[1300:1310])        # 300 -> 310: no group closes
        assert st(cache, [0, 1], s1) == [7, ALL]
        cache.append([0], [0, 108], k[1300:1408], v[1300:1408])       # 1300 -> 1408 closes group 10
        assert st(cache, [0, 1], s1) == [7, ALL]                      # the lowest since the decode
        cache.decode([0, 1], q, 32, out, ws)
        assert st(cache, [0, 1], s1) == [ALL, ALL]
        O_.oscar_cache_reset(cache.handle, 1, s1)
        assert st(cache, [0, 1], s1) == [ALL, 0]
    torch.cuda.synchronize()
    with torch.cuda.stream(s2):
        cache.decode([0], q[:1], 32, out[:1], ws)                     # switch streams
        assert st(cache, [0], s2) == [ALL]
        assert st(cache, [0], s1) == [0]
    torch.cuda.synchronize()
    _check_out(cache, out[:1], q[:1], [0])
    cache.close()


def test_outputs_do_not_depend_on_the_early_copies():
    """Back-to-back decodes (all groups settled), a decode on a fresh stream
    (none), and a decode right after an append that closes groups give the same
    outputs as the oracle over the GPU's cache."""
    O_ = U.lib()
    lens = [5000, 1029, 300]
    cache = O_.OscarCache(3, 8, 8192)
    ks, vs = zip(*[_kv(L + 700, 80 + i) for i, L in enumerate(lens)])
    U.append_all(cache, [0, 1, 2], [k[:L] for k, L in zip(ks, lens)], [v[:L] for v, L in zip(vs, lens)])
    q = W.make_q(3, 32, seed=90).cuda()
    ws = cache.workspace(3, 32)
    outs = [torch.empty((3, 32, 128), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        for o in outs[:3]:
            cache.decode([0, 1, 2], q, 32, o, ws)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    fresh = torch.cuda.Stream()
    with torch.cuda.stream(fresh):
        cache.decode([0, 1, 2], q, 32, outs[3], ws)
    torch.cuda.synchronize()
    assert torch.equal(outs[3], outs[0])
    _check_out(cache, outs[0], q, [0, 1, 2])
    # an append closing groups of every slot, then decodes on the same stream
    with torch.cuda.stream(st):
        U.append_all(cache, [0, 1, 2], [k[L:L + 700] for k, L in zip(ks, lens)],
                     [v[L:L + 700] for v, L in zip(vs, lens)])
        cache.decode([0, 1, 2], q, 32, outs[0], ws)
        cache.decode([0, 1, 2], q, 32, outs[1], ws)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    _check_out(cache, outs[0], q, [0, 1, 2])
    cache.close()


def test_query_written_by_the_preceding_kernel():
    """The kernel right before the decode writes q (as a projection would):
    the decode must read it after its grid dependency wait."""
    O_ = U.lib()
    cache = O_.OscarCache(1, 8, 4096)
    k, v = _kv(3000, 95)
    cache.append([0], [0, 3000], k, v)
    ws = cache.workspace(1, 32)
    st = torch.cuda.Stream()
    n = 1 << 24                                          # a 32 MB bf16 buffer: q is its head
    buf = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    q_true = W.make_q(1, 32, seed=96).cuda()
    add = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    add[:32 * 128] = q_true.reshape(-1)
    out = torch.empty((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    ref = torch.empty_like(out)
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        cache.decode([0], q_true, 32, ref, ws)           # a decode before: blocks are settled
        for step in range(3):
            buf.zero_()
            torch.add(buf, add, out=buf)                  # the preceding kernel writes q
            cache.decode([0], buf[:32 * 128].view(1, 32, 128), 32, out, ws)
            torch.cuda.current_stream().synchronize()
            assert torch.equal(out, ref), f"step {step}: decode read q before the kernel that wrote it finished"
    _check_out(cache, out, q_true, [0])
    cache.close()
