"""GPU parity of the float16-metadata layout (meta_bits = 16).

Quantise: the stored scales, zeros and norms are float16 roundings of float32
values that the GPU and the oracle compute with different rounding orders
(k_hat in float32 against float64; a float32 division against a float64 one
rounded twice), so they agree exactly except where the two float32 values
straddle a float16 rounding boundary: each must lie within one float16 ulp of
the oracle's.  Codes are then checked against the oracle's decision taken with
the GPU's stored parameters, under the boundary rule.  Decode, prefill and the
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
    n_bad = n_tot = 0
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
        # codes: the oracle's decision with the GPU's stored parameters
        kg = U.f64(ks[0][:, h])[: ng * 128].reshape(ng, 128, 128)
        _, k_hat = O.omni_token_scaling(O.canalized_rotation(kg))
        codes, pre = O.int2_codes(k_hat, g.keys.scale[:, None, :], g.keys.zero[:, None, :])
        b, n = P.assert_codes(g.keys.codes, codes, pre, f"K codes head {h}")
        n_bad += b
        n_tot += n
        vg = U.f64(vs[0][:, h])[: ng * 128].reshape(ng, 128, 4, 32)
        codes, pre = O.int2_codes(vg, g.values.scale[..., None], g.values.zero[..., None])
        b, n = P.assert_codes(g.values.codes, codes.reshape(ng, 128, 128), pre.reshape(ng, 128, 128),
                              f"V codes head {h}")
        n_bad += b
        n_tot += n
        assert np.array_equal(g.window_k, r.window_k) and np.array_equal(g.window_v, r.window_v)
    assert n_bad <= P.MAX_BOUNDARY_RATE * n_tot
    print(f"meta16 quantise: {straddles}/{n_params} parameters one float16 ulp from the oracle; "
          f"{n_bad}/{n_tot} boundary code mismatches")


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
