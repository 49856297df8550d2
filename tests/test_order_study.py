"""Pins of the key-path order study (oracle-side analysis, CPU only)."""
import numpy as np

from oracle import oscar_oracle as O
from oracle import order_study as S


def test_exact_inputs_reconstruct_exactly():
    """Keys whose rotated, normalised form is one-hot (rows = column j of the
    unnormalised Hadamard matrix, times a norm: every channel then holds only
    0 and 1, codes 0 and 3) quantise without error through the method's
    pipeline; keys that already sit on 4 equally spaced levels per channel
    (extremes present) quantise without error per channel."""
    Hu = O.hadamard_unnormalised(128)
    rng = np.random.default_rng(0)
    cols = rng.integers(0, 128, size=128)
    norms = 2.0 ** rng.integers(-3, 4, size=128)
    k = Hu[:, cols].T * norms[:, None]        # [128 tokens, 128]
    kh = S.dequantised_keys(k, "rotate_then_scale")
    # exact up to the float32 storage of s (1/3 is not a float32: code 3 gives 1 + 3e-8)
    assert np.max(np.abs(kh - k)) <= 2.0 ** -22 * np.max(np.abs(k))

    levels = rng.integers(0, 4, size=(128, 128)).astype(np.float64)
    levels[0, :] = 0.0
    levels[1, :] = 3.0
    step = 2.0 ** rng.integers(-2, 2, size=128)
    base = rng.integers(-8, 8, size=128) * 0.25
    k2 = base[None, :] + levels * step[None, :]
    kh2 = S.dequantised_keys(k2, "per_channel_only")
    assert np.array_equal(kh2, k2)


def test_orders_agree_up_to_rounding():
    """Scaling by a per-token scalar commutes with the rotation, so the two
    orders quantise the same values up to float64 rounding."""
    rng = np.random.default_rng(1)
    k = rng.standard_normal((512, 128)) * np.exp(0.5 * rng.standard_normal((512, 1)))
    a = S.dequantised_keys(k, "rotate_then_scale")
    b = S.dequantised_keys(k, "scale_then_rotate")
    diff = np.linalg.norm(a - b, axis=-1) / np.linalg.norm(k, axis=-1)
    assert np.mean(diff > 1e-9) <= 1e-2


def test_scaling_protects_small_norm_tokens():
    """A token 1000x smaller than the others: per-channel steps are set by the
    large tokens, so without per-token scaling its relative error is huge;
    with scaling it is quantised on the same footing as the rest."""
    rng = np.random.default_rng(2)
    k = rng.standard_normal((128, 128))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    k[5] *= 1e-3
    sinks = S.sink_mask(k)
    assert sinks.sum() == 1 and sinks[5]
    errs = {name: S.key_errors(k, S.dequantised_keys(k, name), sinks) for name in S.VARIANTS}
    for name in ("rotate_only", "per_channel_only"):
        assert errs[name]["sink_key_rel_err"] > 50.0
    for name in ("rotate_then_scale", "scale_then_rotate", "scale_only"):
        assert errs[name]["sink_key_rel_err"] < 1.0
        assert abs(errs[name]["sink_key_rel_err"] - errs[name]["key_rel_err"]) < 0.5


def test_report_runs():
    rep = S.study(L=512, hkv=1, gqa=2, seed=4)
    assert set(rep) == set(S.VARIANTS)
    for r in rep.values():
        assert r["n_sinks"] >= 1
        assert all(np.isfinite(v) for v in r.values())
    txt = S.format_report(rep)
    assert "rotate_then_scale" in txt
