"""GPU parity of oscar_prefill_attention (a chunk's queries against every token
already in the cache).

Gate, per (query, head) row, against the oracle's history_attention over the
SAME cache read back from the GPU: the output within 2e-3 + half a bf16 ulp
(the decode rule), the log-sum-exp within 1e-3 (score errors of the hi + lo
products are ~1e-6 relative; ex2.approx adds ~2^-22).
"""
import numpy as np
import pytest
import torch

from int2_kv_cache_oscar_gb300 import workloads as W
from oracle import oscar_oracle as O
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu

LSE_TOL = 1e-3


def _run(L, hkv, hq, n_q, seed, scale=0.0, split=False, kvq=None):
    O_ = U.lib()
    gen = torch.Generator().manual_seed(seed)
    k, v = W.make_sequence_kv(L, hkv, W.LLAMA_RECIPE, gen)
    q = torch.randn((n_q, hq, 128), generator=gen).to(torch.bfloat16)
    if kvq is not None:
        k, v, q = kvq(k, v, q)
    cache = O_.OscarCache(1, hkv, L + 128)
    U.append_all(cache, [0], [k], [v])
    out = torch.empty((n_q, hq, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((n_q, hq), dtype=torch.float32, device="cuda")
    ws = None
    if split:
        nb = O_.oscar_prefill_workspace_bytes(cache.handle, 0, n_q, hq)
        assert nb > 0, "expected a split history"
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    O_.oscar_prefill_attention(cache.handle, 0, q.cuda(), hq, scale, out, lse, workspace=ws)
    torch.cuda.synchronize()
    O_.oscar_cache_check(cache.handle)
    arena = U.read_arena(cache)
    got, gl, qn = U.f64(out), lse.cpu().numpy().astype(np.float64), U.f64(q)
    gqa = hq // hkv
    worst = worst_lse = 0.0
    for j in range(hkv):
        head = U.gpu_head(cache, arena, 0, j)
        rows = qn[:, j * gqa:(j + 1) * gqa].reshape(-1, 128)      # query-major rows
        o_ref, l_ref = O.history_attention(rows, head, None if scale == 0.0 else scale)
        o_gpu = got[:, j * gqa:(j + 1) * gqa].reshape(-1, 128)
        l_gpu = gl[:, j * gqa:(j + 1) * gqa].reshape(-1)
        worst = max(worst, P.assert_decode(o_gpu, o_ref, f"L={L} head {j}"))
        e = float(np.abs(l_gpu - l_ref).max())
        assert e <= LSE_TOL, f"L={L} head {j}: lse error {e:.2e}"
        worst_lse = max(worst_lse, e)
    print(f"prefill L={L} hkv={hkv} hq={hq} n_q={n_q} split={split}: max|o err|={worst:.2e} "
          f"max|lse err|={worst_lse:.2e}")
    return out, lse


@pytest.mark.parametrize("L", [8192 + 100, 8192, 2048 + 1])
def test_prefill_split_history(L):
    """With a workspace the history is split into parts (separate CTAs) and
    merged; the rows still meet the oracle's rule, and agree with the unsplit
    call within rounding (the merge changes only the summation order)."""
    o1, l1 = _run(L, hkv=2, hq=8, n_q=37, seed=91, split=True)
    o0, l0 = _run(L, hkv=2, hq=8, n_q=37, seed=91)
    a, b = o1.float(), o0.float()
    assert bool(((a - b).abs() <= 2e-3 + b.abs() * 2.0 ** -7).all())     # within one bf16 ulp (+ 2e-3)
    assert float((l1 - l0).abs().max()) <= 1e-4


def test_prefill_workspace_too_small_runs_unsplit():
    O_ = U.lib()
    gen = torch.Generator().manual_seed(95)
    k, v = W.make_sequence_kv(4096, 2, W.LLAMA_RECIPE, gen)
    cache = O_.OscarCache(1, 2, 4096)
    U.append_all(cache, [0], [k], [v])
    q = torch.randn((5, 8, 128), generator=gen).to(torch.bfloat16).cuda()
    nb = O_.oscar_prefill_workspace_bytes(cache.handle, 0, 5, 8)
    assert nb > 0
    out_a, out_b = torch.empty_like(q), torch.empty_like(q)
    O_.oscar_prefill_attention(cache.handle, 0, q, 8, 0.0, out_a)
    one_part = 2 * 5 * 4 * 528                       # Hkv x rows x a 528-byte record
    small = torch.empty(one_part + 16, dtype=torch.uint8, device="cuda")   # room for one part, not two
    O_.oscar_prefill_attention(cache.handle, 0, q, 8, 0.0, out_b, workspace=small)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    with pytest.raises(O_.OscarError):      # host memory is not a workspace
        O_.oscar_prefill_attention(cache.handle, 0, q, 8, 0.0, out_b,
                                   workspace=torch.empty(nb, dtype=torch.uint8).pin_memory())


@pytest.mark.parametrize("L", [8192 + 100, 1024, 100, 129, 1])
def test_prefill_history_lengths(L):
    _run(L, hkv=2, hq=8, n_q=37, seed=61 + L % 7)


@pytest.mark.parametrize("gqa", [1, 2, 3, 4, 6])
def test_prefill_gqa(gqa):
    _run(2048 + 17, hkv=2, hq=2 * gqa, n_q=20, seed=70 + gqa)


def test_prefill_scale_and_single_query():
    _run(4096 + 5, hkv=1, hq=4, n_q=1, seed=80, scale=0.05)


def test_prefill_bad_args():
    O_ = U.lib()
    cache = O_.OscarCache(2, 2, 256)
    q = torch.zeros((3, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(O_.OscarError) as e:
        O_.oscar_prefill_attention(cache.handle, 0, q, 8, 0.0, out)     # empty sequence
    assert e.value.status == O_.OSCAR_ERR_INVALID_ARG
    k = torch.zeros((10, 2, 128), dtype=torch.bfloat16, device="cuda")
    cache.append([0], [0, 10], k, k)
    q7 = torch.zeros((3, 7, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(O_.OscarError) as e:
        O_.oscar_prefill_attention(cache.handle, 0, q7, 7, 0.0, torch.empty_like(q7))  # heads not a multiple of Hkv
    assert e.value.status == O_.OSCAR_ERR_INVALID_ARG
    with pytest.raises(O_.OscarError) as e:
        O_.oscar_prefill_attention(cache.handle, 5, q, 8, 0.0, out)     # slot out of range
    assert e.value.status == O_.OSCAR_ERR_INVALID_ARG


def test_prefill_gqa8():
    """8 query heads per KV head (rows = queries x 8 per KV head)."""
    _run(2048 + 40, hkv=2, hq=16, n_q=11, seed=97)


def _bf16(x):
    return x.to(torch.bfloat16)


# inputs that stretch the operand scalings: value zeros far above the value
# scales, of both signs (the zero sums accumulate across groups in one
# per-CTA unit); window keys up to ~1e4 (the rotated keys' fp16 pieces carry
# 2^fw) and down to ~1e-4 (queries scaled the other way, so that scores stay
# moderate); scores that grow along the sequence (the running maximum moves
# by more than 8 in log2 units several times, so O and the zero sums are
# rescaled in TMEM)
_EXTREME = {
    "value_offset": lambda k, v, q: (k, _bf16(v.float() * 0.02 + torch.where(
        (torch.arange(v.shape[0]) // 128 % 2 == 0)[:, None, None], 40.0, -25.0)), q),
    "large_window_keys": lambda k, v, q: (_bf16(k.float() * 700.0), v, _bf16(q.float() / 700.0)),
    "small_window_keys": lambda k, v, q: (_bf16(k.float() * 1e-4), v, _bf16(q.float() * 1e4)),
    "growing_scores": lambda k, v, q: (_bf16(k.float() * torch.linspace(0.05, 4.0, k.shape[0])[:, None, None]), v, q),
}


@pytest.mark.parametrize("case", sorted(_EXTREME))
def test_prefill_extreme_magnitudes(case):
    _run(2048 + 100, hkv=2, hq=8, n_q=33, seed=101, kvq=_EXTREME[case])
    _run(2048 + 100, hkv=2, hq=8, n_q=33, seed=101, kvq=_EXTREME[case], split=True)
