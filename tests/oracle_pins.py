"""Pins of the CPU oracle against facts fixed by mathematics and by the pages.

Each check returns None when the oracle satisfies it and a message string when
it does not, so that the same checks serve the plain pin tests and the
mutation tests (which plant a mistake in the oracle and expect a check to
fail).

What fixes each check:
* the Sylvester Hadamard construction (textbook recursion, scipy.linalg's
  routine, a hand-typed H_8) and its algebra (orthogonality, symmetry, the
  all-ones vector, energy spreading of a spike, norm preservation);
* the norm identity k = n * H^T k_hat of Omni-Token Scaling;
* hand-derived worked examples of the asymmetric INT2 quantiser, one of
  them with quotients a hair off a tie;
* closed forms: keys that are scaled Hadamard columns rotate to one-hot
  vectors, so their codes, scales and norms are known exactly;
* losslessness on inputs already on the 4 levels;
* the quantiser error bound |x - x_hat| <= s / 2;
* brute-force attention written with explicit Python loops;
* attention special cases (one token, zero query, one dominant score,
  window only, lossless keys reduce to exact attention, GQA mapping).
"""
from __future__ import annotations

import math
import os

import numpy as np

from oracle import oscar_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D = 128


def _load_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return np.array(rows)


def _bf16(x):
    """Round float64 values to bf16 (round to nearest even) and back."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- Hadamard

def check_hadamard_scipy():
    import scipy.linalg
    H = O.hadamard(D)
    ref = scipy.linalg.hadamard(D).astype(np.float64) / math.sqrt(D)
    if not np.array_equal(H, ref):
        return "H_d differs from scipy.linalg.hadamard(d)/sqrt(d)"


def check_hadamard_golden8():
    H8 = _load_golden("hadamard8_sylvester.txt")
    if not np.array_equal(O.hadamard(8) * math.sqrt(8), H8):
        return "H_8 differs from the hand-typed Sylvester matrix"


def check_hadamard_algebra():
    H = O.hadamard(D)
    if np.abs(H @ H.T - np.eye(D)).max() > 1e-14:
        return "H H^T != I"
    if not np.array_equal(H, H.T):
        return "H not symmetric"
    ones = np.ones(D)
    e0 = np.zeros(D)
    e0[0] = math.sqrt(D)
    if np.abs(O.canalized_rotation(ones) - e0).max() > 1e-12:
        return "H 1 != sqrt(d) e_0"


def check_energy_spreading():
    # a x20 spike in one channel spreads to magnitude 20/sqrt(d) everywhere
    for c in (3, 77):
        x = np.zeros(D)
        x[c] = 20.0
        r = O.canalized_rotation(x)
        if np.abs(np.abs(r) - 20.0 / math.sqrt(D)).max() > 1e-12:
            return f"spike at channel {c} not spread uniformly"
        # sign pattern is column c of the unnormalised matrix
        if not np.array_equal(np.sign(r), np.sign(O.hadamard(D)[:, c])):
            return "spike signs differ from Hadamard column"


def check_norm_preserved():
    rng = np.random.default_rng(11)
    k = rng.standard_normal((64, D)) * rng.lognormal(0, 1, (64, 1))
    r = O.canalized_rotation(k)
    if np.abs(np.linalg.norm(r, axis=1) / np.linalg.norm(k, axis=1) - 1).max() > 1e-13:
        return "rotation changes norms"


# ------------------------------------------------------- Omni-Token Scaling

def check_norm_identity():
    rng = np.random.default_rng(12)
    k = _bf16(rng.standard_normal((128, D)) * 3.0)
    k[5] = 0.0
    g = O.quantize_key_group(k)
    r = O.canalized_rotation(k)
    n, k_hat = O.omni_token_scaling(r)
    if np.abs(np.linalg.norm(k_hat[np.arange(128) != 5], axis=1) - 1).max() > 1e-13:
        return "k_hat not unit norm"
    if np.any(k_hat[5] != 0.0) or n[5] != 0.0:
        return "zero key does not map to zero"
    back = n[:, None] * (k_hat @ O.hadamard(D))        # n H^T k_hat (row form)
    if np.abs(back - k).max() > 1e-12 * np.abs(k).max():
        return "k != n H^T k_hat"
    if np.abs(g.norm.astype(np.float64) - np.linalg.norm(k, axis=1)).max() > \
            1e-6 * np.linalg.norm(k, axis=1).max():
        return "stored norm != L2 norm of the key"


# ------------------------------------------------------------- quantiser

def check_worked_example():
    t = _load_golden("int2_asym_worked.txt")
    x = t[:, 0]
    g = O.quantize_value_group(np.tile(x, 4)[None, :])   # one token, 4 equal groups
    if not np.allclose(g.scale, 1.0) or not np.allclose(g.zero, -1.0):
        return f"worked example s/z wrong: {g.scale} {g.zero}"
    codes = g.codes[0, :32]
    if not np.array_equal(codes, t[:, 2].astype(np.uint8)):
        return f"worked example codes wrong: {codes} vs {t[:, 2]}"
    if not np.array_equal(g.pre[0, :32], t[:, 1]):
        return "worked example pre-rounding values wrong"
    if not np.array_equal(O.dequant_values(g)[0, :32], t[:, 3]):
        return "worked example dequantised values wrong"


def check_near_tie_example():
    """Hand-derived near-tie example (tests/golden/int2_asym_near_tie.txt):
    the code follows the exact (x - z) / s of the stored float32 scale, also
    where a float32 evaluation of that quotient lands on a tie."""
    from fractions import Fraction
    rows = []
    with open(os.path.join(GOLDEN, "int2_asym_near_tie.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                g, x, num, den, code = line.split()
                rows.append((g, float(x), Fraction(int(num), int(den)), int(code)))
    names = ["A", "B", "C", "A"]
    x = np.zeros((1, D))
    for gi, name in enumerate(names):
        vals = [r[1] for r in rows if r[0] == name]
        x[0, 32 * gi:32 * gi + 32] = [vals[i % len(vals)] for i in range(32)]
    g = O.quantize_value_group(x)
    want_s = {"A": np.float32(11184811 / 2 ** 25), "B": np.float32(41943039 / (3 * 2 ** 25)),
              "C": np.float32(0.5)}
    for gi, name in enumerate(names):
        if g.scale[0, gi] != want_s[name]:
            return f"near-tie example: group {name} scale {g.scale[0, gi]!r}"
        vals = [r for r in rows if r[0] == name]
        for i in range(32):
            _, xv, pre, code = vals[i % len(vals)]
            if g.codes[0, 32 * gi + i] != code:
                return f"near-tie example: group {name} x = {xv} code {g.codes[0, 32 * gi + i]} != {code}"
            if abs(Fraction(float(g.pre[0, 32 * gi + i])) - pre) > Fraction(1, 2 ** 50) * max(pre, 1):
                return f"near-tie example: group {name} x = {xv} pre-rounding value wrong"


def check_value_lossless():
    rng = np.random.default_rng(13)
    T = 128
    z = rng.integers(-64, 64, (T, 4)) / 16.0
    s = 2.0 ** rng.integers(-4, 3, (T, 4))
    c = rng.integers(0, 4, (T, 4, 32))
    c[:, :, 0] = 0
    c[:, :, 1] = 3                                   # both extremes present
    x = (z[..., None] + s[..., None] * c).reshape(T, D)
    g = O.quantize_value_group(x)
    if not np.array_equal(g.codes.reshape(T, 4, 32), c.astype(np.uint8)):
        return "value codes not recovered on exact levels"
    if not np.array_equal(O.dequant_values(g), x):
        return "value round trip not exact on exact levels"
    if not (np.array_equal(g.scale, s.astype(np.float32)) and
            np.array_equal(g.zero, z.astype(np.float32))):
        return "value scale/zero not exact"


def check_key_onehot_closed_form():
    """k_t = a_t * (column pi(t) of the unnormalised Hadamard matrix), a_t > 0.
    Then H_d k_t = a_t sqrt(d) e_pi(t): n_t = a_t sqrt(d), k_hat_t = e_pi(t).
    Per channel c: values are 1 on tokens with pi(t) = c, else 0, so
    s_c = 1/3 (float32), z_c = 0, code = 3 there and 0 elsewhere; channels no
    token maps to have s = 0 and all codes 0."""
    rng = np.random.default_rng(14)
    Hu = np.round(O.hadamard(D) * math.sqrt(D))
    pi = rng.integers(0, D, 128)
    a = 2.0 ** rng.integers(-3, 4, 128)
    k = a[:, None] * Hu[:, pi].T
    g = O.quantize_key_group(k)
    exp_codes = np.zeros((128, D), np.uint8)
    exp_codes[np.arange(128), pi] = 3
    if not np.array_equal(g.codes, exp_codes):
        return "one-hot key codes wrong"
    used = np.zeros(D, bool)
    used[pi] = True
    exp_s = np.where(used, np.float32(1.0 / 3.0), np.float32(0.0))
    if not (np.array_equal(g.scale, exp_s) and np.array_equal(g.zero, np.zeros(D, np.float32))):
        return "one-hot key scale/zero wrong"
    if not np.array_equal(g.norm, (a * math.sqrt(D)).astype(np.float32)):
        return "one-hot key norms wrong"


def check_error_bound():
    rng = np.random.default_rng(15)
    k = _bf16(rng.standard_normal((3, 128, D)) * np.array([1, 10, 0.01])[:, None, None])
    g = O.quantize_key_group(k)
    r = O.canalized_rotation(k)
    _, k_hat = O.omni_token_scaling(r)
    err = np.abs(O.dequant_keys(g) - k_hat)
    bound = g.scale.astype(np.float64)[:, None, :] / 2 + 4e-7
    if np.any(err > bound):
        return "key quantisation error exceeds s/2"
    v = _bf16(rng.standard_normal((3, 128, D)) * 5)
    gv = O.quantize_value_group(v)
    errv = np.abs(O.dequant_values(gv) - v).reshape(3, 128, 4, 32)
    bv = gv.scale.astype(np.float64)[..., None] / 2 + 4e-7 * np.abs(v).max()
    if np.any(errv > bv):
        return "value quantisation error exceeds s/2"


def check_constant_channel():
    rng = np.random.default_rng(16)
    v = rng.standard_normal((128, D))
    v[:, 32:64] = 0.75                                 # one constant value group
    g = O.quantize_value_group(v)
    if not (np.all(g.scale[:, 1] == 0) and np.all(g.codes[:, 32:64] == 0)):
        return "constant group: s != 0 or codes != 0"
    if not np.all(O.dequant_values(g)[:, 32:64] == 0.75):
        return "constant group: dequant != z"


def check_group_alignment():
    rng = np.random.default_rng(17)
    L = 300
    k = _bf16(rng.standard_normal((L, D)))
    v = _bf16(rng.standard_normal((L, D)))
    c = O.build_head_cache(k, v)
    if c.num_groups != 2 or c.window_k.shape[0] != 44:
        return "wrong group / window split"
    g1 = O.quantize_key_group(k[128:256])
    if not (np.array_equal(c.keys.codes[1], g1.codes) and np.array_equal(c.keys.scale[1], g1.scale)):
        return "group 1 is not quantised from positions 128..255 alone"
    if not np.array_equal(c.window_v, v[256:]):
        return "window is not the raw tail"


# ------------------------------------------------------------- attention

def _brute_decode(q, cache, scale):
    """Explicit loops: dequantise every token, score, softmax, weighted sum."""
    H = O.hadamard(D)
    Hg = q.shape[0]
    out = np.zeros((Hg, D))
    for h in range(Hg):
        qr = [sum(H[i][j] * q[h][j] for j in range(D)) for i in range(D)]
        scores, vals = [], []
        for g in range(cache.num_groups):
            for t in range(128):
                acc = 0.0
                for c in range(D):
                    kh = float(cache.keys.codes[g, t, c]) * float(cache.keys.scale[g, c]) \
                        + float(cache.keys.zero[g, c])
                    acc += qr[c] * kh
                scores.append(float(cache.keys.norm[g, t]) * acc * scale)
                row = []
                for c in range(D):
                    gi = c // 32
                    row.append(float(cache.values.codes[g, t, c]) * float(cache.values.scale[g, t, gi])
                               + float(cache.values.zero[g, t, gi]))
                vals.append(row)
        for t in range(cache.window_k.shape[0]):
            scores.append(sum(q[h][c] * cache.window_k[t][c] for c in range(D)) * scale)
            vals.append(list(cache.window_v[t]))
        m = max(scores)
        w = [math.exp(s - m) for s in scores]
        tot = sum(w)
        for c in range(D):
            out[h][c] = sum(w[t] * vals[t][c] for t in range(len(w))) / tot
    return out


def check_brute_force_attention():
    rng = np.random.default_rng(18)
    L = 131
    k = _bf16(rng.standard_normal((L, D)) * 2)
    v = _bf16(rng.standard_normal((L, D)))
    q = _bf16(rng.standard_normal((2, D)))
    c = O.build_head_cache(k, v)
    scale = 1 / math.sqrt(D)
    got = O.decode_head(q, c, scale)
    ref = _brute_decode(q, c, scale)
    if np.abs(got - ref).max() > 1e-12:
        return f"decode differs from brute force by {np.abs(got - ref).max()}"


def check_single_token():
    rng = np.random.default_rng(19)
    k = _bf16(rng.standard_normal((1, D)))
    v = _bf16(rng.standard_normal((1, D)))
    c = O.build_head_cache(k, v)
    o = O.decode_head(_bf16(rng.standard_normal((3, D))), c)
    if not np.array_equal(o, np.repeat(v, 3, axis=0)):
        return "L=1 output != v_0"


def check_zero_query_mean():
    rng = np.random.default_rng(20)
    L = 256 + 17
    k = _bf16(rng.standard_normal((L, D)))
    v = _bf16(rng.standard_normal((L, D)))
    c = O.build_head_cache(k, v)
    o = O.decode_head(np.zeros((1, D)), c)
    mean = O.decode_values(c).mean(axis=0)
    if np.abs(o[0] - mean).max() > 1e-13:
        return "q = 0 output != mean of dequantised values"


def check_dominant_score():
    """Keys are scaled one-hot Hadamard columns; the query points along one of
    them with a huge norm, so one score exceeds the rest by > 700 and its
    value row is returned (also exercises max subtraction: scores ~ 1e3)."""
    Hu = np.round(O.hadamard(D) * math.sqrt(D))
    L = 128
    pi = np.arange(L) % D
    k = Hu[:, pi].T.copy()
    rng = np.random.default_rng(21)
    v = _bf16(rng.standard_normal((L, D)))
    q = np.zeros((1, D))
    q[0] = Hu[:, 7] * 1.0                    # q . k_t = 128 for t = 7, else 0
    c = O.build_head_cache(k, v)
    o = O.decode_head(q * 60.0, c, softmax_scale=1.0)
    vd = O.decode_values(c)
    if not np.all(np.isfinite(o)) or np.abs(o[0] - vd[7]).max() > 1e-12:
        return "dominant score does not return its value row"


def check_window_only_exact():
    rng = np.random.default_rng(22)
    L = 100
    k = _bf16(rng.standard_normal((L, D)))
    v = _bf16(rng.standard_normal((L, D)))
    q = _bf16(rng.standard_normal((4, D)))
    c = O.build_head_cache(k, v)
    if np.abs(O.decode_head(q, c) - O.attention_exact(q, k, v)).max() > 1e-14:
        return "window-only decode != exact attention"


def check_lossless_keys_exact():
    """Keys = a_t * Hadamard column with a_t a power of two, values on exact
    levels: the cache is lossless up to float32 s = 1/3, so decode must
    equal unquantised attention; this fixes the n_t factor, the rotation of q
    and the scale."""
    rng = np.random.default_rng(23)
    Hu = np.round(O.hadamard(D) * math.sqrt(D))
    L = 256 + 9
    pi = rng.integers(0, D, L)
    a = 2.0 ** rng.integers(-6, -2, L)
    k = a[:, None] * Hu[:, pi].T
    k[256:] = _bf16(rng.standard_normal((9, D)))
    lv = rng.integers(0, 4, (L, 4, 32)).astype(np.float64)
    lv[:, :, 0], lv[:, :, 1] = 0, 3
    v = (lv * 0.25 - 0.5).reshape(L, D)
    q = _bf16(rng.standard_normal((4, D)))
    c = O.build_head_cache(k, v)
    got = O.decode_head(q, c)
    ref = O.attention_exact(q, k, v)
    if np.abs(got - ref).max() > 1e-6:
        return f"lossless cache decode != exact attention ({np.abs(got - ref).max()})"


def check_gqa_mapping():
    """Hq = 4, Hkv = 2: query head h must read KV head h // 2."""
    rng = np.random.default_rng(24)
    L = 40
    ks = [_bf16(rng.standard_normal((L, D))) for _ in range(2)]
    vs = [_bf16(rng.standard_normal((L, D))) for _ in range(2)]
    q = _bf16(rng.standard_normal((1, 4, D)))
    caches = [[O.build_head_cache(ks[j], vs[j]) for j in range(2)]]
    out = O.decode_attention(q, caches)
    for h in range(4):
        ref = O.attention_exact(q[0, h:h + 1], ks[h // 2], vs[h // 2])
        if np.abs(out[0, h] - ref[0]).max() > 1e-14:
            return f"query head {h} does not read KV head {h // 2}"


ALL_CHECKS = [
    check_hadamard_scipy, check_hadamard_golden8, check_hadamard_algebra,
    check_energy_spreading, check_norm_preserved, check_norm_identity,
    check_worked_example, check_near_tie_example, check_value_lossless, check_key_onehot_closed_form,
    check_error_bound, check_constant_channel, check_group_alignment,
    check_brute_force_attention, check_single_token, check_zero_query_mean,
    check_dominant_score, check_window_only_exact, check_lossless_keys_exact,
    check_gqa_mapping,
]
