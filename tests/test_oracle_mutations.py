"""Plant plausible mistakes in the oracle (on the CPU) and check that the pin
suite notices each one.  This shows that the pins constrain every step of
the oracle: rotation, norm scaling, quantiser parameters, rounding, grouping,
dequantisation, the decode score, softmax and the GQA mapping."""
import numpy as np
import pytest

from oracle import oscar_oracle as O
from tests import oracle_pins as P

_orig = {name: getattr(O, name) for name in dir(O) if callable(getattr(O, name))}


def _hadamard_flip(d=128):
    H = _orig["hadamard_unnormalised"](d).copy()
    H[3, 5] = -H[3, 5]
    return H


def _hadamard_sequency(d=128):
    H = _orig["hadamard_unnormalised"](d)
    sign_changes = (np.diff(H, axis=1) != 0).sum(axis=1)
    return H[np.argsort(sign_changes, kind="stable")]


def _rotation_unnormalised(k):
    return k @ _orig["hadamard_unnormalised"](k.shape[-1]).T


def _scaling_no_divide(r):
    n = np.sqrt(np.sum(r * r, axis=-1))
    return n, r


def _params_div4(x_min, x_max):
    return ((x_max - x_min) / 4).astype(np.float32), np.asarray(x_min).astype(np.float32)


def _codes_floor(x, s32, z32):
    codes, pre = _orig["int2_codes"](x, s32, z32)
    return np.clip(np.floor(pre), 0, 3).astype(np.uint8), pre


def _codes_half_up(x, s32, z32):
    codes, pre = _orig["int2_codes"](x, s32, z32)
    return np.clip(np.floor(pre + 0.5), 0, 3).astype(np.uint8), pre


def _codes_fp32_reciprocal(x, s32, z32):
    """The decision taken in float32 as fl32(fl32(x - z) * fl32(1 / s))."""
    x32 = np.asarray(x, np.float64).astype(np.float32)
    s = np.asarray(s32, np.float32)
    z = np.asarray(z32, np.float32)
    ok = s > 0
    inv = np.where(ok, np.float32(1) / np.where(ok, s, np.float32(1)), np.float32(0)).astype(np.float32)
    pre = ((x32 - z).astype(np.float32) * inv).astype(np.float32)
    return np.clip(np.rint(pre), 0, 3).astype(np.uint8), pre.astype(np.float64)


def _codes_fp32_division(x, s32, z32):
    """The decision taken in float32 as fl32(fl32(x - z) / s)."""
    x32 = np.asarray(x, np.float64).astype(np.float32)
    s = np.asarray(s32, np.float32)
    z = np.asarray(z32, np.float32)
    ok = s > 0
    pre = np.where(ok, (x32 - z).astype(np.float32) / np.where(ok, s, np.float32(1)), np.float32(0))
    pre = pre.astype(np.float32)
    return np.clip(np.rint(pre), 0, 3).astype(np.uint8), pre.astype(np.float64)


def _dequant_no_zero(codes, s32, z32):
    return codes.astype(np.float64) * np.asarray(s32, np.float64)


def _key_group_channel_axis(k):
    k = np.asarray(k, dtype=np.float64)
    n, k_hat = O.omni_token_scaling(O.canalized_rotation(k))
    s32, z32 = O.int2_params(k_hat.min(axis=-1), k_hat.max(axis=-1))   # wrong axis
    codes, pre = O.int2_codes(k_hat, s32[..., None], z32[..., None])
    return O.KeyGroup(codes, s32, z32, n.astype(np.float32), pre)


def _scores_no_norm(q, cache, softmax_scale=None):
    q = np.asarray(q, dtype=np.float64)
    scale = (1.0 / np.sqrt(q.shape[-1])) if softmax_scale is None else softmax_scale
    parts = []
    if cache.num_groups > 0:
        k_hat = O.dequant_keys(cache.keys).reshape(-1, q.shape[-1])
        parts.append((k_hat @ O.canalized_rotation(q).T) * scale)
    if cache.window_k.shape[0] > 0:
        parts.append((cache.window_k @ q.T) * scale)
    return np.concatenate(parts, axis=0)


def _scores_unrotated_q(q, cache, softmax_scale=None):
    q = np.asarray(q, dtype=np.float64)
    scale = (1.0 / np.sqrt(q.shape[-1])) if softmax_scale is None else softmax_scale
    parts = []
    if cache.num_groups > 0:
        k_hat = O.dequant_keys(cache.keys).reshape(-1, q.shape[-1])
        n = cache.keys.norm.astype(np.float64).reshape(-1)
        parts.append((k_hat @ q.T) * n[:, None] * scale)
    if cache.window_k.shape[0] > 0:
        parts.append((cache.window_k @ q.T) * scale)
    return np.concatenate(parts, axis=0)


def _scores_window_rotated(q, cache, softmax_scale=None):
    q = np.asarray(q, dtype=np.float64)
    scale = (1.0 / np.sqrt(q.shape[-1])) if softmax_scale is None else softmax_scale
    parts = []
    if cache.num_groups > 0:
        k_hat = O.dequant_keys(cache.keys).reshape(-1, q.shape[-1])
        n = cache.keys.norm.astype(np.float64).reshape(-1)
        parts.append((k_hat @ O.canalized_rotation(q).T) * n[:, None] * scale)
    if cache.window_k.shape[0] > 0:
        parts.append((cache.window_k @ O.canalized_rotation(q).T) * scale)
    return np.concatenate(parts, axis=0)


def _softmax_no_max(scores, values):
    with np.errstate(over="ignore", invalid="ignore"):
        e = np.exp(scores)
        p = e / e.sum(axis=0, keepdims=True)
    return p.T @ values


def _decode_attention_wrong_gqa(q, caches, softmax_scale=None):
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    out = np.zeros((B, Hq, d))
    for b in range(B):
        Hkv = len(caches[b])
        for h in range(Hq):
            out[b, h] = O.decode_head(q[b, h:h + 1], caches[b][h % Hkv], softmax_scale)[0]
    return out


MUTATIONS = {
    "hadamard_sign_flip": ("hadamard_unnormalised", _hadamard_flip),
    "hadamard_sequency_order": ("hadamard_unnormalised", _hadamard_sequency),
    "rotation_unnormalised": ("canalized_rotation", _rotation_unnormalised),
    "scaling_without_divide": ("omni_token_scaling", _scaling_no_divide),
    "scale_over_4_levels": ("int2_params", _params_div4),
    "codes_floor": ("int2_codes", _codes_floor),
    "codes_round_half_up": ("int2_codes", _codes_half_up),
    "codes_fp32_reciprocal": ("int2_codes", _codes_fp32_reciprocal),
    "codes_fp32_division": ("int2_codes", _codes_fp32_division),
    "dequant_drops_zero": ("int2_dequant", _dequant_no_zero),
    "key_params_wrong_axis": ("quantize_key_group", _key_group_channel_axis),
    "score_drops_norm": ("decode_scores", _scores_no_norm),
    "score_unrotated_query": ("decode_scores", _scores_unrotated_q),
    "window_rotated_query": ("decode_scores", _scores_window_rotated),
    "softmax_no_max_subtraction": ("softmax_attend", _softmax_no_max),
    "gqa_modulo_mapping": ("decode_attention", _decode_attention_wrong_gqa),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    failures = []
    for check in P.ALL_CHECKS:
        try:
            msg = check()
        except Exception as e:  # a crash also counts as detection
            msg = f"raised {type(e).__name__}"
        if msg is not None:
            failures.append(check.__name__)
    assert failures, f"mutation {name} passed every pin"


def test_value_group_width_mutation(monkeypatch):
    monkeypatch.setattr(O, "VALUE_GROUP", 16)
    msgs = [c() for c in (P.check_worked_example, P.check_value_lossless)]
    assert any(m is not None for m in msgs)
