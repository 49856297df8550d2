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
