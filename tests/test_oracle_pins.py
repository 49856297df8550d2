"""The CPU oracle against closed forms, invariants, a worked example and brute
force (see tests/oracle_pins.py for what fixes each check)."""
import pytest

from tests import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    msg = check()
    assert msg is None, msg


def test_history_attention_lse_and_merge():
    """lse of all-equal scores over T tokens is ln T plus the score; the
    log-sum-exp merge of two disjoint key sets equals attention over their
    union (window-only caches hold the keys exactly)."""
    import numpy as np

    from oracle import oscar_oracle as O

    rng = np.random.default_rng(11)
    d = 128
    k = rng.standard_normal((100, d))
    v = rng.standard_normal((100, d))
    q0 = np.zeros((3, d))
    # window-only caches (fewer than 128 tokens are never quantised)
    full = O.build_head_cache(k, v)
    o, lse = O.history_attention(q0, full)
    assert np.allclose(lse, np.log(100.0), atol=1e-12)
    assert np.allclose(o, v.mean(axis=0)[None, :], atol=1e-12)
    q = rng.standard_normal((5, d))
    o_all, lse_all = O.history_attention(q, full)
    a = O.build_head_cache(k[:37], v[:37])
    b = O.build_head_cache(k[37:], v[37:])
    o1, l1 = O.history_attention(q, a)
    o2, l2 = O.history_attention(q, b)
    om, lm = O.merge_attention(o1, l1, o2, l2)
    assert np.allclose(om, o_all, atol=1e-12) and np.allclose(lm, lse_all, atol=1e-12)
    # brute force: lse = ln sum exp(q.k / sqrt(d))
    s = (k @ q.T) / np.sqrt(d)
    assert np.allclose(lse_all, np.log(np.exp(s).sum(axis=0)), atol=1e-10)


def test_fp16_metadata_quantiser():
    """16-bit metadata layout: values on 4 levels with float16-exact scale
    and zero round-trip exactly; on random data the reconstruction error is
    bounded by half a step plus the float16 rounding of s and z (the codes
    are decided against the rounded parameters, with clamping)."""
    import numpy as np

    from oracle import oscar_oracle as O

    rng = np.random.default_rng(12)
    levels = rng.integers(0, 4, size=(64, 128)).astype(np.float64)
    levels[:, 0] = 0.0
    levels[:, 1] = 3.0                       # both extremes in every 32-channel group
    levels[:, 32] = 0.0
    levels[:, 33] = 3.0
    levels[:, 64] = 0.0
    levels[:, 65] = 3.0
    levels[:, 96] = 0.0
    levels[:, 97] = 3.0
    v = -1.5 + 0.25 * levels                  # z = -1.5, s = 0.25: exact in float16
    g = O.quantize_value_group(v, meta_bits=16)
    assert np.array_equal(O.dequant_values(g), v)
    assert g.scale.dtype == np.float32 and np.all(g.scale == 0.25) and np.all(g.zero == -1.5)

    x = rng.standard_normal((64, 128)) * 3.0
    g = O.quantize_value_group(x, meta_bits=16)
    xr = x.reshape(64, 4, 32)
    m, M = xr.min(axis=-1), xr.max(axis=-1)
    s_true = (M - m) / 3
    err = np.abs(O.dequant_values(g).reshape(64, 4, 32) - xr)
    bound = g.scale / 2 + np.abs(g.zero - m) + 3 * np.abs(g.scale - s_true) + 1e-6 * np.abs(m)
    assert np.all(err <= bound[..., None] + 1e-12)
    # float16 rounding actually happened (the layout is not a float32 copy)
    assert np.all(g.scale == g.scale.astype(np.float16).astype(np.float32))
    assert np.any(g.scale != s_true.astype(np.float32))
    kg = O.quantize_key_group(x.reshape(1, 64, 128)[:, :64], meta_bits=16)
    assert np.all(kg.norm == kg.norm.astype(np.float16).astype(np.float32))
