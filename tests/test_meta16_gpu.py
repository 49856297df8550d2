"""GPU parity of the float16-metadata layout (meta_bits = 16).

Quantise: the stored scales, zeros and norms are float16 roundings of float32
values that the GPU and the oracle compute with different rounding orders
(k_hat in float32 against float64; a float32 division against a float64 one
rounded twice), so they agree exactly except where the two float32 values
straddle a float16 rounding boundary: each must lie within one float16 ulp of
the oracle's.  Codes are checked against the oracle's own decision (its own
float16 parameters) under the boundary rule; a mismatch is excused only where
the code was decided against a parameter that differs by that ulp, and those
are counted apart.  Decode, prefill and the
fused step are checked against the oracle over the GPU's own cache, with the
decode rule.
"""
import numpy as np
import pytest
import torch

from int2_kv_cache_oscar_gb300 import workloads as W
from oracle import oscar_oracle as O
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu


def _f16_ulp(x):
    x = np.abs(np.asarray(x, np.float32)).astype(np.float16)
    return (np.nextafter(x, np.float16(np.inf)) - x).astype(np.float64)


def _cache(lens, hkv, seed, chunk=None, max_len=None):
    gen = torch.Generator().manual_seed(seed)
    ks, vs = [], []
    for L in lens:
        k, v = W.make_sequence_kv(L, hkv, W.LLAMA_RECIPE, gen)
        ks.append(k)
        vs.append(v)
    c = U.lib().OscarCache(len(lens), hkv, max_len or max(lens) + 128, meta_bits=16)
    U.append_all(c, list(range(len(lens))), ks, vs, chunk=chunk)
    return c, ks, vs


@pytest.mark.parametrize("chunk", [None, 1000])
def test_meta16_quantize_parity(chunk):
    c, ks, vs = _cache([8192 + 100], 8, seed=91, chunk=chunk)
    arena = U.read_arena(c)
    straddles = n_params = 0
    counts = {"K": [0, 0, 0], "V": [0, 0, 0]}     # boundary mismatches, excused mismatches, codes
    for h in range(8):
        g = U.gpu_head(c, arena, 0, h)
        r = U.oracle_head(ks[0], vs[0], h, meta_bits=16)
        ng = g.num_groups
        assert ng == r.num_groups
        for what, gv, rv in [("K scale", g.keys.scale, r.keys.scale), ("K zero", g.keys.zero, r.keys.zero),
                             ("K norm", g.keys.norm, r.keys.norm), ("V scale", g.values.scale, r.values.scale),
                             ("V zero", g.values.zero, r.values.zero)]:
            d = np.abs(gv.astype(np.float64) - rv.astype(np.float64))
            assert np.all(d <= _f16_ulp(rv) * 1.0001), f"{what} head {h}: more than one float16 ulp apart"
            straddles += int(np.count_nonzero(d))
            n_params += d.size
        # codes: the oracle's own decision (its own float16 parameters).  A
        # mismatch is excused only where the code was decided against a
        # parameter whose stored float16 differs between the two sides (the
        # one-ulp straddles counted above), and is otherwise held to the
        # boundary rule.
        k_diff = (g.keys.scale != r.keys.scale) | (g.keys.zero != r.keys.zero)          # [ng, 128 channels]
        v_diff = (g.values.scale != r.values.scale) | (g.values.zero != r.values.zero)  # [ng, 128 tokens, 4]
        cases = (("K", g.keys.codes, r.keys, np.broadcast_to(k_diff[:, None, :], g.keys.codes.shape)),
                 ("V", g.values.codes, r.values, np.repeat(v_diff, 32, axis=-1)))
        for name, gc, rc, excused in cases:
            b, n = P.assert_codes(gc, rc.codes, rc.pre, f"{name} codes head {h}", excused=excused)
            counts[name][0] += b
            counts[name][1] += int(np.count_nonzero((gc != rc.codes) & excused))
            counts[name][2] += n
        assert np.array_equal(g.window_k, r.window_k) and np.array_equal(g.window_v, r.window_v)
    for name, (b, e, n) in counts.items():
        assert b <= P.MAX_BOUNDARY_RATE * n, f"{name}: boundary mismatch rate {b}/{n}"
        print(f"meta16 quantise {name}: {b}/{n} boundary code mismatches; {e} mismatches where a stored "
              f"parameter differs by one float16 ulp")
    print(f"meta16 quantise: {straddles}/{n_params} parameters one float16 ulp from the oracle")


def test_meta16_chunking_is_bit_identical():
    states = []
    for chunk in [None, 7, 129]:
        c, _, _ = _cache([700], 8, seed=92, chunk=chunk, max_len=1024)
        states.append(U.live_bytes(c, U.read_arena(c), 0))
    for st in states[1:]:
        assert np.array_equal(st, states[0])


@pytest.mark.parametrize("lens", [[8192 + 37], [300, 5000, 129]])
def test_meta16_decode_parity(lens):
    c, ks, vs = _cache(lens, 8, seed=93)
    hq = 32
    q = W.make_q(len(lens), hq, seed=94)
    out = torch.empty((len(lens), hq, 128), dtype=torch.bfloat16, device="cuda")
    ws = c.workspace(len(lens), hq)
    c.decode(list(range(len(lens))), q.cuda(), hq, out, ws)
    U.lib().oscar_cache_check(c.handle)
    arena = U.read_arena(c)
    got, qn = U.f64(out), U.f64(q)
    worst = 0.0
    for i in range(len(lens)):
        for j in range(8):
            ref = O.decode_head(qn[i, 4 * j:4 * j + 4], U.gpu_head(c, arena, i, j))
            worst = max(worst, P.assert_decode(got[i, 4 * j:4 * j + 4], ref, f"seq {i} head {j}"))
    print(f"meta16 decode {lens}: max|gpu - oracle(gpu cache)| = {worst:.2e}")


def test_meta16_prefill_and_fused_step():
    O_ = U.lib()
    c, ks, vs = _cache([2048 + 50], 2, seed=95)
    hq, n_q = 8, 21
    gen = torch.Generator().manual_seed(96)
    q = torch.randn((n_q, hq, 128), generator=gen).to(torch.bfloat16)
    out = torch.empty((n_q, hq, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((n_q, hq), dtype=torch.float32, device="cuda")
    arena = U.read_arena(c)
    qn = U.f64(q)
    nb = O_.oscar_prefill_workspace_bytes(c.handle, 0, n_q, hq)
    assert nb > 0                                   # 16 groups: the history splits
    for ws in (None, torch.empty(nb, dtype=torch.uint8, device="cuda")):
        O_.oscar_prefill_attention(c.handle, 0, q.cuda(), hq, 0.0, out, lse, workspace=ws)
        got, gl = U.f64(out), lse.cpu().numpy()
        for j in range(2):
            rows = qn[:, 4 * j:4 * j + 4].reshape(-1, 128)
            o_ref, l_ref = O.history_attention(rows, U.gpu_head(c, arena, 0, j))
            P.assert_decode(got[:, 4 * j:4 * j + 4].reshape(-1, 128), o_ref, f"prefill head {j} split {ws is not None}")
            assert np.abs(gl[:, 4 * j:4 * j + 4].reshape(-1) - l_ref).max() <= 1e-3
    # fused decode step against separate calls on a twin cache
    c2, _, _ = _cache([2048 + 50], 2, seed=95)
    kn = torch.randn((1, 2, 128), generator=gen).to(torch.bfloat16).cuda()
    vn = torch.randn((1, 2, 128), generator=gen).to(torch.bfloat16).cuda()
    q1 = torch.randn((1, hq, 128), generator=gen).to(torch.bfloat16).cuda()
    o1 = torch.empty((1, hq, 128), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    c.append([0], [0, 1], kn, vn)
    c.decode([0], q1, hq, o1, c.workspace(1, hq))
    c2.append_decode([0], kn, vn, q1, hq, o2, c2.workspace(1, hq))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
