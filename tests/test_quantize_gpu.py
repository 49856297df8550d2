"""GPU parity of the compression path (oscar_quantize_append) against the CPU
oracle: codes bit-exact except inside the 1e-3 boundary window (rate
<= 1e-5), scales / zeros / norms within 1e-6 relative, window bytes exact."""
import numpy as np
import pytest
import torch

from int2_kv_cache_oscar_gb300 import workloads as W
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu


def _compare_cache(cache, slots, ks, vs, report):
    arena = U.read_arena(cache)
    counts = {"K": [0, 0], "V": [0, 0]}
    worst = {"kscale": 0.0, "kzero": 0.0, "knorm": 0.0, "vscale": 0.0, "vzero": 0.0}
    for i, s in enumerate(slots):
        L = ks[i].shape[0]
        assert cache.length(s) == L
        for h in range(ks[i].shape[1]):
            g = U.gpu_head(cache, arena, s, h)
            r = U.oracle_head(ks[i], vs[i], h)
            assert g.num_groups == r.num_groups
            if r.num_groups:
                for name, gc, rc in (("K", g.keys, r.keys), ("V", g.values, r.values)):
                    b, n = P.assert_codes(gc.codes, rc.codes, rc.pre, f"{name} codes slot {s} head {h}")
                    counts[name][0] += b
                    counts[name][1] += n
                worst["kscale"] = max(worst["kscale"], P.assert_meta(g.keys.scale, r.keys.scale, "K scale"))
                worst["kzero"] = max(worst["kzero"], P.assert_meta(g.keys.zero, r.keys.zero, "K zero"))
                worst["knorm"] = max(worst["knorm"], P.assert_meta(g.keys.norm, r.keys.norm, "K norm"))
                worst["vscale"] = max(worst["vscale"], P.assert_meta(g.values.scale, r.values.scale, "V scale"))
                worst["vzero"] = max(worst["vzero"], P.assert_meta(g.values.zero, r.values.zero, "V zero"))
            assert np.array_equal(g.window_k, r.window_k) and np.array_equal(g.window_v, r.window_v)
    for name, (n_bad, n_tot) in counts.items():
        assert n_bad <= P.MAX_BOUNDARY_RATE * max(n_tot, 1), f"{name} boundary mismatch rate {n_bad}/{n_tot}"
        report[f"{name}_code_mismatch"] = (n_bad, n_tot)
    report.update(worst)
    return report


def test_tiny_layer_parity():
    """1 KV head, d=128, 1024 tokens = 8 full groups; channels 3, 77 x20; sink."""
    w = W.tiny_layer()
    ks, vs, _ = W.make_workload_tensors(w)
    O_ = U.lib()
    cache = O_.OscarCache(1, 1, 1024)
    U.append_all(cache, [0], ks, vs)
    rep = _compare_cache(cache, [0], ks, vs, {})
    print("tiny layer", rep)


@pytest.mark.parametrize("chunk", [None, 4096, 1000])
def test_llama_layer_with_window(chunk):
    """32/8 heads, 8192 + 100 tokens (64 groups + a 100-token window per head)."""
    w = W.llama_layer(8192 + 100)
    ks, vs, _ = W.make_workload_tensors(w)
    O_ = U.lib()
    cache = O_.OscarCache(1, 8, 8192 + 256)
    U.append_all(cache, [0], ks, vs, chunk=chunk)
    rep = _compare_cache(cache, [0], ks, vs, {})
    print("llama layer", chunk, rep)


def test_chunking_is_bit_identical():
    """Appending the same tokens at once, in odd chunks, or one at a time
    (closing groups mid-stream from window + new tokens) gives identical
    arenas."""
    w = W.llama_layer(700, seed=9)
    ks, vs, _ = W.make_workload_tensors(w)
    O_ = U.lib()
    states = []
    for chunk in [None, 1, 7, 100, 129, lambda i, p: 1 + (p * 7919) % 200]:
        cache = O_.OscarCache(2, 8, 1024)
        U.append_all(cache, [1], ks, vs, chunk=chunk)
        states.append(U.live_bytes(cache, U.read_arena(cache), 1))
    for st in states[1:]:
        assert np.array_equal(st, states[0])


def test_ragged_batch_append():
    """Several sequences of different lengths appended in the same calls with
    different chunkings; slots not in order."""
    lens = [1, 127, 128, 129, 300, 1000]
    gen = torch.Generator().manual_seed(11)
    ks, vs = [], []
    for L in lens:
        k, v = W.make_sequence_kv(L, 8, W.LLAMA_RECIPE, gen)
        ks.append(k)
        vs.append(v)
    slots = [5, 0, 3, 1, 4, 2]
    O_ = U.lib()
    cache = O_.OscarCache(6, 8, 1024)
    U.append_all(cache, slots, ks, vs, chunk=lambda i, p: [1, 50, 128, 200, 33, 77][i])
    _compare_cache(cache, slots, ks, vs, {})


def test_capacity_and_bad_args_leave_state():
    O_ = U.lib()
    cache = O_.OscarCache(2, 8, 256)
    gen = torch.Generator().manual_seed(3)
    k, v = W.make_sequence_kv(200, 8, W.LLAMA_RECIPE, gen)
    U.append_all(cache, [0], [k], [v])
    before = U.read_arena(cache)
    kk, vv = k[:100].cuda(), v[:100].cuda()
    with pytest.raises(O_.OscarError) as e:
        cache.append([0], [0, 100], kk, vv)                 # 300 > 256
    assert e.value.status == O_.OSCAR_ERR_CAPACITY
    with pytest.raises(O_.OscarError):
        cache.append([0, 0], [0, 1, 2], kk, vv)             # repeated slot
    with pytest.raises(O_.OscarError):
        cache.append([2], [0, 1], kk, vv)                   # slot out of range
    with pytest.raises(O_.OscarError):
        cache.append([1], [1, 2], kk, vv)                   # cu_new[0] != 0
    assert cache.length(0) == 200 and cache.length(1) == 0
    assert np.array_equal(U.read_arena(cache), before)


def test_cache_bytes():
    O_ = U.lib()
    cache = O_.OscarCache(3, 8, 2048)
    gen = torch.Generator().manual_seed(4)
    lens = {0: 1000, 2: 256}
    for s, L in lens.items():
        k, v = W.make_sequence_kv(L, 8, W.LLAMA_RECIPE, gen)
        U.append_all(cache, [s], [k], [v])
    used = O_.oscar_cache_bytes(cache.handle, -1, O_.OSCAR_BYTES_USED)
    bf16 = O_.oscar_cache_bytes(cache.handle, -1, O_.OSCAR_BYTES_BF16_EQUIVALENT)
    exp_used = sum(8 * ((L // 128) * 13824 + (L % 128) * 512) for L in lens.values())
    assert used == exp_used
    assert bf16 == sum(8 * L * 512 for L in lens.values())
    assert O_.oscar_cache_bytes(cache.handle, 2, O_.OSCAR_BYTES_USED) == 8 * 2 * 13824
    # full groups: 65536 / 13824 = 4.74x smaller than bf16
    assert abs(65536 / 13824 - 4.7407) < 1e-3


def test_16_byte_aligned_inputs_match_32_byte_aligned():
    """Inputs that are 16- but not 32-byte aligned take the 16-byte row loads
    (the 32-byte loads need 32-byte alignment); the arena must be identical
    to the one built from 32-byte aligned inputs, windows and a group closed
    from window + new rows included."""
    w = W.llama_layer(2 * 128 + 90, seed=21)
    ks, vs, _ = W.make_workload_tensors(w)
    k, v = ks[0], vs[0]
    O_ = U.lib()
    states = []
    for offset in (0, 8):                     # bf16 elements: 0 or 16 bytes past a 256-byte boundary
        cache = O_.OscarCache(1, 8, 1024)
        for p0, n in ((0, 100), (100, 200), (300, 46)):
            bk = torch.empty(n * 8 * 128 + offset, dtype=torch.bfloat16, device="cuda")
            bv = torch.empty_like(bk)
            kk = bk[offset:].view(n, 8, 128)
            vv = bv[offset:].view(n, 8, 128)
            kk.copy_(k[p0:p0 + n])
            vv.copy_(v[p0:p0 + n])
            assert (kk.data_ptr() % 32 == 0) == (offset == 0) and kk.data_ptr() % 16 == 0
            cache.append([0], [0, n], kk, vv)
        O_.oscar_cache_check(cache.handle)
        states.append(U.live_bytes(cache, U.read_arena(cache), 0))
    assert np.array_equal(states[0], states[1])
    cache = O_.OscarCache(1, 8, 1024)
    U.append_all(cache, [0], ks, vs, chunk=100)
    _compare_cache(cache, [0], ks, vs, {})


@pytest.mark.parametrize("meta_bits", [32, 16])
def test_header_maxima(meta_bits):
    """The arena header's per-(slot, head) maxima (include/oscar.h): the
    largest stored value scale and the largest |stored value zero| over the
    quantised groups, exactly; both equal the oracle's within its parameter
    tolerance; a reset of the slot clears them, and appends after it start
    over."""
    gen = torch.Generator().manual_seed(71)
    hkv, slots = 4, 3
    lens = [1000, 300, 128 * 5]
    ks, vs = [], []
    for L in lens:
        k, v = W.make_sequence_kv(L, hkv, W.LLAMA_RECIPE, gen)
        ks.append(k)
        vs.append(v)
    cache = U.lib().OscarCache(slots, hkv, 1024, meta_bits=meta_bits)
    U.append_all(cache, list(range(slots)), ks, vs, chunk=333)

    def header(arena):
        words = arena[256:256 + 2 * slots * hkv * 4].view(np.float32)
        return words[:slots * hkv].reshape(slots, hkv), words[slots * hkv:].reshape(slots, hkv)

    arena = U.read_arena(cache)
    smax, zmax = header(arena)
    for s in range(slots):
        for h in range(hkv):
            g = U.gpu_head(cache, arena, s, h)
            r = U.oracle_head(ks[s], vs[s], h, meta_bits=meta_bits)
            assert smax[s, h] == np.float32(np.max(g.values.scale)), f"slot {s} head {h}: value-scale maximum"
            assert zmax[s, h] == np.float32(np.max(np.abs(g.values.zero))), f"slot {s} head {h}: |zero| maximum"
            tol = 1e-6 if meta_bits == 32 else 2.0 ** -10
            assert abs(smax[s, h] - np.max(r.values.scale)) <= tol * np.max(r.values.scale)
            assert abs(zmax[s, h] - np.max(np.abs(r.values.zero))) <= tol * np.max(np.abs(r.values.zero))
    # a reset clears the slot's maxima; the next append records its own
    U.lib().oscar_cache_reset(cache.handle, 1)
    k2, v2 = W.make_sequence_kv(256, hkv, W.LLAMA_RECIPE, gen)
    v2 = (v2.float() * 0.01).to(torch.bfloat16)     # far smaller values: the new maxima must drop
    arena_before = header(U.read_arena(cache))
    assert np.all(arena_before[0][1] == 0) and np.all(arena_before[1][1] == 0)
    U.append_all(cache, [1], [k2], [v2])
    arena = U.read_arena(cache)
    smax, zmax = header(arena)
    for h in range(hkv):
        g = U.gpu_head(cache, arena, 1, h)
        assert smax[1, h] == np.float32(np.max(g.values.scale))
        assert zmax[1, h] == np.float32(np.max(np.abs(g.values.zero)))
