"""GPU compression against closed forms, and degenerate inputs.

The rotation is the normalised Sylvester Hadamard matrix H_d = Hu / sqrt(128),
Hu[i][j] = (-1)^popcount(i & j) (OScaR abstract; ai-papers.net "OScaRの提案手法":
Canalized Rotation, then Omni-Token Scaling, then per-channel INT2).

* Keys whose rows are columns pi(t) of Hu (entries +-1, exact in bf16):
  Hu k = 128 e_pi(t) exactly, so the norm is sqrt(128^2 / 128) = sqrt(128),
  k_hat = e_pi(t), every channel holds one 1 and 127 zeros over the group:
  scale fl32(1/3), zero 0, code 3 at channel pi(t) and 0 elsewhere.  Pins
  the transform's order and normalisation and the packing of key codes.
* Keys whose rows are basis vectors e_pi(t): k_hat = Hu e_pi(t) / sqrt(128),
  norm 1; channel 0 is constant (+1/sqrt(128), scale 0, code 0), every other
  channel splits evenly between +-1/sqrt(128): code 3 where
  Hu[c][pi(t)] = +1, else 0.
* Values on 4 dyadic levels z + s * code per token and 32-channel group, both
  extremes present: codes, s and z come back exactly.
The first two tests use no oracle; the degenerate-input case (zero-norm
tokens, an all-zero key group, an all-zero value group) and key tokens whose
squares under- or overflow float32 are checked against it.
"""
import numpy as np
import pytest
import torch

from tests import gpu_util as U

pytestmark = pytest.mark.gpu

D = G = 128


def _sylvester():
    i = np.arange(D)
    pc = np.vectorize(lambda x: bin(x).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0)


def _values(rng, hkv):
    """[G, hkv, D] values z + s * code with s = 0.25, z = -1.5 and both extreme
    levels in every 32-channel group of every token; returns (v, codes)."""
    codes = rng.integers(0, 4, size=(G, hkv, D))
    for gr in range(4):
        codes[:, :, 32 * gr] = 0
        codes[:, :, 32 * gr + 1] = 3
    return -1.5 + 0.25 * codes, codes


def _run(keys, values, hkv):
    cache = U.lib().OscarCache(1, hkv, G)
    k = torch.tensor(keys, dtype=torch.float32).to(torch.bfloat16)
    v = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(k.double(), torch.tensor(keys)) and torch.equal(v.double(), torch.tensor(values))
    cache.append([0], [0, G], k.cuda(), v.cuda())
    U.lib().oscar_cache_check(cache.handle)
    arena = U.read_arena(cache)
    return [U.gpu_head(cache, arena, 0, h) for h in range(hkv)]


def _check_values(g, vcodes):
    assert np.array_equal(g.values.codes[0], vcodes)
    assert np.all(g.values.scale[0] == np.float32(0.25)) and np.all(g.values.zero[0] == np.float32(-1.5))


def test_hadamard_columns_give_one_hot_codes():
    rng = np.random.default_rng(11)
    hkv = 2
    Hu = _sylvester()
    perms = [rng.permutation(D) for _ in range(hkv)]
    keys = np.stack([Hu[:, perms[h]].T for h in range(hkv)], axis=1)   # [t, h, c] = Hu[c][pi_h(t)]
    values, vcodes = _values(rng, hkv)
    heads = _run(keys, values, hkv)
    for h, g in enumerate(heads):
        expect = np.zeros((G, D), np.uint8)
        expect[np.arange(G), perms[h]] = 3
        assert np.array_equal(g.keys.codes[0], expect), f"head {h}: key codes"
        assert np.all(g.keys.scale[0] == np.float32(1.0) / np.float32(3.0)), f"head {h}: key scales"
        assert np.all(g.keys.zero[0] == 0.0), f"head {h}: key zeros"
        assert np.all(g.keys.norm[0] == np.sqrt(np.float32(128.0))), f"head {h}: norms"
        _check_values(g, vcodes[:, h])


def test_basis_vectors_give_hadamard_sign_codes():
    rng = np.random.default_rng(12)
    hkv = 2
    Hu = _sylvester()
    perms = [rng.permutation(D) for _ in range(hkv)]
    keys = np.zeros((G, hkv, D))
    for h in range(hkv):
        keys[np.arange(G), h, perms[h]] = 1.0
    values, vcodes = _values(rng, hkv)
    heads = _run(keys, values, hkv)
    r = np.float32(1.0) / np.sqrt(np.float32(128.0))          # 1 / sqrt(128), as float32
    for h, g in enumerate(heads):
        cols = Hu[:, perms[h]].T                                # [t, c] = Hu[c][pi(t)]
        expect = np.where(cols > 0, 3, 0).astype(np.uint8)
        expect[:, 0] = 0                                        # channel 0: constant, scale 0
        assert np.array_equal(g.keys.codes[0], expect), f"head {h}: key codes"
        assert np.all(g.keys.norm[0] == 1.0), f"head {h}: norms"
        assert g.keys.scale[0][0] == 0.0 and g.keys.zero[0][0] == r
        s = (np.float32(2.0) * r) / np.float32(3.0)
        assert np.all(np.abs(g.keys.scale[0][1:] - s) <= 1e-6 * s), f"head {h}: key scales"
        assert np.all(np.abs(g.keys.zero[0][1:] + r) <= 1e-6 * r), f"head {h}: key zeros"
        _check_values(g, vcodes[:, h])


def test_zero_norm_tokens_and_constant_channels():
    """Degenerate inputs: all-zero key tokens (norm 0, k_hat = 0: score 0,
    still in the softmax), a whole group of zero keys (every rotated channel
    constant: scale 0, codes 0), and a 32-channel value group that is zero in
    every token of a group (scale 0, zero 0, codes 0); quantisation and decode
    against the oracle, the zero tokens' norms exactly 0."""
    from int2_kv_cache_oscar_gb300 import workloads as W
    from oracle import oscar_oracle as O
    from tests import parity as P

    gen = torch.Generator().manual_seed(13)
    L, hkv, hq = 3 * G + 40, 2, 8
    k, v = W.make_sequence_kv(L, hkv, W.LLAMA_RECIPE, gen)
    zero_tok = [5, 77, 128 + 3, 300, 3 * G + 7]
    k[zero_tok] = 0
    k[G:2 * G, 0, :] = 0                 # head 0: group 1 entirely zero
    v[:G, 1, 32:64] = 0                  # head 1: value group 1 zero across tokens of group 0
    cache = U.lib().OscarCache(1, hkv, L + 8)
    U.append_all(cache, [0], [k], [v], chunk=100)
    q = W.make_q(1, hq, seed=14)
    out = torch.empty((1, hq, 128), dtype=torch.bfloat16, device="cuda")
    cache.decode([0], q.cuda(), hq, out, cache.workspace(1, hq))
    U.lib().oscar_cache_check(cache.handle)
    arena = U.read_arena(cache)
    got, qn = U.f64(out), U.f64(q)
    for h in range(hkv):
        g = U.gpu_head(cache, arena, 0, h)
        r = U.oracle_head(k, v, h)
        P.assert_codes(g.keys.codes, r.keys.codes, r.keys.pre, f"head {h} K codes")
        P.assert_codes(g.values.codes, r.values.codes, r.values.pre, f"head {h} V codes")
        for name in ("scale", "zero", "norm"):
            P.assert_meta(getattr(g.keys, name), getattr(r.keys, name), f"head {h} K {name}")
        norms = g.keys.norm.reshape(-1)
        for t in zero_tok:
            if t < 3 * G:
                assert norms[t] == 0.0, f"head {h}: token {t} norm {norms[t]}"
        P.assert_decode(got[0, 4 * h:4 * h + 4], O.decode_head(qn[0, 4 * h:4 * h + 4], g), f"head {h} decode")
    g0 = U.gpu_head(cache, arena, 0, 0)
    assert np.all(g0.keys.norm[1] == 0) and np.all(g0.keys.scale[1] == 0) and np.all(g0.keys.codes[1] == 0)
    g1 = U.gpu_head(cache, arena, 0, 1)
    assert np.all(g1.values.scale[0][:, 1] == 0) and np.all(g1.values.zero[0][:, 1] == 0)
    assert np.all(g1.values.codes[0][:, 32:64] == 0)


def test_extreme_key_norms():
    """Key tokens whose squared channels under- or overflow float32: tokens
    near 1e-24 and 1e-30, a token at the bf16 subnormal level, and tokens
    near 1e22 (squares above 1e38).  Norms, scales, zeros and codes against
    the oracle, and the decode over the GPU's cache (the huge tokens dominate
    the softmax)."""
    from int2_kv_cache_oscar_gb300 import workloads as W
    from oracle import oscar_oracle as O
    from tests import parity as P

    gen = torch.Generator().manual_seed(17)
    L, hkv, hq = 2 * G + 30, 2, 8
    k, v = W.make_sequence_kv(L, hkv, W.LLAMA_RECIPE, gen)
    k = k.double()
    scale = {3: 1e-24, 40: 1e-30, 77: 1e-24, 90: 1e22, G + 5: 1e-40, G + 60: 1e22, G + 61: 1e-24}
    for t, f in scale.items():
        k[t] *= f
    k = k.to(torch.bfloat16)
    assert torch.isfinite(k.float()).all() and 0 < k[G + 5].float().abs().max() < 1.18e-38
    cache = U.lib().OscarCache(1, hkv, L + 8)
    U.append_all(cache, [0], [k], [v])
    q = W.make_q(1, hq, seed=18)
    out = torch.empty((1, hq, 128), dtype=torch.bfloat16, device="cuda")
    cache.decode([0], q.cuda(), hq, out, cache.workspace(1, hq))
    U.lib().oscar_cache_check(cache.handle)
    arena = U.read_arena(cache)
    got, qn = U.f64(out), U.f64(q)
    for h in range(hkv):
        g = U.gpu_head(cache, arena, 0, h)
        r = U.oracle_head(k, v, h)
        P.assert_codes(g.keys.codes, r.keys.codes, r.keys.pre, f"head {h} K codes")
        for name in ("scale", "zero", "norm"):
            P.assert_meta(getattr(g.keys, name), getattr(r.keys, name), f"head {h} K {name}")
        norms = g.keys.norm.reshape(-1)
        for t in scale:
            assert norms[t] > 0.0 and np.isfinite(norms[t]), f"head {h}: token {t} norm {norms[t]}"
        P.assert_decode(got[0, 4 * h:4 * h + 4], O.decode_head(qn[0, 4 * h:4 * h + 4], g), f"head {h} decode")
