"""Parity at the full sizes of the benchmark workloads, built and decoded in
the launch configuration bench.py times, on samples the oracle computes one
by one:

* 128K-token sequence, 32 query / 8 KV heads, the whole prefill in one
  append, one decode call: the decode output of two KV heads against the
  oracle over the GPU's cache of those heads (the decode rule), and the codes
  and parameters of every group of those heads against the oracle's
  quantisation of the same tokens (the code and metadata rules, the
  boundary-mismatch rate taken over all codes the test compares);
* batch 32 x 32K tokens (sinks at 1 % of positions), one decode call over
  the batch: three sequences, one KV head each, the same checks;
* ragged serving stream, 8 sequences of 4K..128K tokens, prefill in
  4096-token chunks, then 256 single-token steps (separate append and
  decode calls, then the fused call), so that groups close mid-stream and
  the window rolls over: decode of the last step and every group (those
  closed during the stream included), for two sampled sequences.

* chunked prefill, 512 queries x 32 heads against a 32K-token history with
  the library's workspace (the history split into parts, then the merge):
  24 sampled queries of two KV heads.

The error against unquantised attention of the sampled heads is printed.
"""
import numpy as np
import pytest
import torch

from int2_kv_cache_oscar_gb300 import workloads as W
from oracle import oscar_oracle as O
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu

HKV, HQ = 8, 32


def _gen(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


def _check_groups(g_head, k_tok, v_tok, what):
    """Codes and parameters of every GPU group of one head against the
    oracle's quantisation of the same tokens (k_tok, v_tok: float64 [L, 128]).
    A mismatch outside the boundary window fails here; returns the boundary
    mismatches and the codes compared, for the rate over the whole test."""
    ng = g_head.num_groups
    kk = k_tok[:128 * ng].reshape(ng, 128, 128)
    vv = v_tok[:128 * ng].reshape(ng, 128, 128)
    rk, rv = O.quantize_key_group(kk), O.quantize_value_group(vv)
    counts = {}
    for name, gc, rc in (("K", g_head.keys.codes, rk), ("V", g_head.values.codes, rv)):
        b, n_out, n = P.code_mismatches(gc, rc.codes, rc.pre)
        assert n_out == 0, f"{what}: {n_out} {name} code mismatches outside the boundary window"
        counts[name] = np.array([b, n])
    P.assert_meta(g_head.keys.scale, rk.scale, f"{what} K scale")
    P.assert_meta(g_head.keys.zero, rk.zero, f"{what} K zero")
    P.assert_meta(g_head.keys.norm, rk.norm, f"{what} K norm")
    P.assert_meta(g_head.values.scale, rv.scale, f"{what} V scale")
    P.assert_meta(g_head.values.zero, rv.zero, f"{what} V zero")
    return counts


def _add(acc, counts):
    for name, c in counts.items():
        acc[name] = acc.get(name, 0) + c
    return acc


def _rate_ok(acc, what):
    for name, (n_bad, n_tot) in sorted(acc.items()):
        assert n_bad <= P.MAX_BOUNDARY_RATE * n_tot, f"{what}: {name} boundary mismatch rate {n_bad}/{n_tot}"
        print(f"{what}: {name} codes {n_bad}/{n_tot} boundary mismatches (rate {n_bad / n_tot:.2e})")


def _check_decode(got, qn, g_head, k_tok, v_tok, what):
    ref = O.decode_head(qn, g_head)
    worst = P.assert_decode(got, ref, what)
    exact = O.attention_exact(qn, k_tok, v_tok)
    return worst, float(np.abs(got - exact).max())


def test_128k_decode_and_sampled_groups():
    L = 131072
    k, v = W.make_sequence_kv(L, HKV, W.LLAMA_RECIPE, _gen(2), "cuda")
    q = W.make_q(1, HQ, seed=2, device="cuda")
    cache = U.lib().OscarCache(1, HKV, L)
    cache.append([0], [0, L], k, v)
    out = torch.empty((1, HQ, 128), dtype=torch.bfloat16, device="cuda")
    cache.decode([0], q, HQ, out, cache.workspace(1, HQ))
    U.lib().oscar_cache_check(cache.handle)
    arena = U.read_arena(cache)
    got, qn = U.f64(out), U.f64(q)
    acc = {}
    for head in (0, 5):
        g = U.gpu_head(cache, arena, 0, head)
        assert g.num_groups == 1024 and g.window_k.shape[0] == 0
        kt, vt = U.f64(k[:, head]), U.f64(v[:, head])
        _add(acc, _check_groups(g, kt, vt, f"128K head {head}"))
        worst, exact = _check_decode(got[0, 4 * head:4 * head + 4], qn[0, 4 * head:4 * head + 4], g, kt, vt,
                                     f"128K head {head}")
        print(f"128K head {head}: decode max|gpu - oracle(gpu cache)| = {worst:.2e}, vs unquantised {exact:.2e}")
    _rate_ok(acc, "128K, 2 heads")


def test_batch32_32k_decode_sampled():
    B, L = 32, 32768
    rec = W.multi_batch(B, L).recipe
    gen = _gen(3)
    cache = U.lib().OscarCache(B, HKV, L)
    ks, vs = [], []
    for b in range(B):
        k, v = W.make_sequence_kv(L, HKV, rec, gen, "cuda")
        cache.append([b], [0, L], k, v)
        ks.append(k)
        vs.append(v)
    q = W.make_q(B, HQ, seed=3, device="cuda")
    out = torch.empty((B, HQ, 128), dtype=torch.bfloat16, device="cuda")
    cache.decode(list(range(B)), q, HQ, out, cache.workspace(B, HQ))
    U.lib().oscar_cache_check(cache.handle)
    arena = U.read_arena(cache)
    got, qn = U.f64(out), U.f64(q)
    acc = {}
    for b, head in ((0, 3), (17, 6), (31, 0)):
        g = U.gpu_head(cache, arena, b, head)
        kt, vt = U.f64(ks[b][:, head]), U.f64(vs[b][:, head])
        _add(acc, _check_groups(g, kt, vt, f"batch seq {b} head {head}"))
        worst, exact = _check_decode(got[b, 4 * head:4 * head + 4], qn[b, 4 * head:4 * head + 4], g, kt, vt,
                                     f"batch seq {b} head {head}")
        print(f"batch 32x32K seq {b} head {head}: decode max|gpu - oracle(gpu cache)| = {worst:.2e}, "
              f"vs unquantised {exact:.2e}")
    _rate_ok(acc, "batch 32x32K, 3 heads")


def test_ragged_stream_sampled():
    lens = W.ragged_lengths(8)
    steps = 256
    gen = _gen(4)
    O_ = U.lib()
    cache = O_.OscarCache(8, HKV, max(lens) + steps)
    ks, vs = [], []
    for i, L in enumerate(lens):
        k, v = W.make_sequence_kv(L, HKV, W.LLAMA_RECIPE, gen, "cuda")
        for p0 in range(0, L, 4096):
            n = min(4096, L - p0)
            cache.append([i], [0, n], k[p0:p0 + n].contiguous(), v[p0:p0 + n].contiguous())
        ks.append(k)
        vs.append(v)
    g2 = _gen(44)
    newk = torch.randn((steps, 8, HKV, 128), generator=g2, device="cuda").to(torch.bfloat16)
    newv = torch.randn((steps, 8, HKV, 128), generator=g2, device="cuda").to(torch.bfloat16)
    q = W.make_q(8, HQ, seed=4, device="cuda")
    out = torch.empty((8, HQ, 128), dtype=torch.bfloat16, device="cuda")
    ws = cache.workspace(8, HQ)
    ids = list(range(8))
    for st in range(steps):
        if st < steps // 2:
            cache.append(ids, list(range(9)), newk[st], newv[st])
            cache.decode(ids, q, HQ, out, ws)
        else:
            cache.append_decode(ids, newk[st], newv[st], q, HQ, out, ws)
    O_.oscar_cache_check(cache.handle)
    arena = U.read_arena(cache)
    got, qn = U.f64(out), U.f64(q)
    acc = {}
    for i, head in ((int(np.argmax(lens)), 2), (int(np.argmin(lens)), 7)):
        L0 = lens[i]
        assert cache.length(i) == L0 + steps
        kt = np.concatenate([U.f64(ks[i][:, head]), U.f64(newk[:, i, head])])
        vt = np.concatenate([U.f64(vs[i][:, head]), U.f64(newv[:, i, head])])
        g = U.gpu_head(cache, arena, i, head)
        closed = list(range(L0 // 128, (L0 + steps) // 128))        # groups closed during the stream
        assert len(closed) >= 2
        _add(acc, _check_groups(g, kt, vt, f"stream seq {i} head {head}"))
        assert np.array_equal(g.window_k, kt[128 * ((L0 + steps) // 128):])
        worst, exact = _check_decode(got[i, 4 * head:4 * head + 4], qn[i, 4 * head:4 * head + 4], g, kt, vt,
                                     f"stream seq {i} head {head}")
        print(f"stream seq {i} (L {L0} + {steps}) head {head}: groups closed {closed}; decode max|gpu - oracle| = "
              f"{worst:.2e}, vs unquantised {exact:.2e}")
    _rate_ok(acc, "stream, 2 heads")


def test_prefill_512x32k_sampled():
    """Chunked prefill at the bench's size and launch configuration: 512
    queries x 32 heads against a 32K-token history, with the workspace the
    library asks for (the history split into parts, then the merge).  Every
    row of two KV heads' sampled queries against the oracle over the GPU's
    cache: the output by the decode rule, the log-sum-exp within 1e-3."""
    O_ = U.lib()
    L, C = 32768, 512
    k, v = W.make_sequence_kv(L, HKV, W.LLAMA_RECIPE, _gen(5), "cuda")
    cache = O_.OscarCache(1, HKV, L)
    cache.append([0], [0, L], k, v)
    q = torch.randn((C, HQ, 128), generator=_gen(55), device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    lse = torch.empty((C, HQ), dtype=torch.float32, device="cuda")
    nb = O_.oscar_prefill_workspace_bytes(cache.handle, 0, C, HQ)
    assert nb > 0, "the bench's configuration splits the history"
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    O_.oscar_prefill_attention(cache.handle, 0, q, HQ, 0.0, out, lse, workspace=ws)
    torch.cuda.synchronize()
    O_.oscar_cache_check(cache.handle)
    arena = U.read_arena(cache)
    gqa = HQ // HKV
    qs = np.random.default_rng(7).choice(C, size=24, replace=False)      # sampled queries
    got, gl, qn = U.f64(out), lse.cpu().numpy().astype(np.float64), U.f64(q)
    for j in (2, 7):
        head = U.gpu_head(cache, arena, 0, j)
        rows = qn[qs, j * gqa:(j + 1) * gqa].reshape(-1, 128)
        o_ref, l_ref = O.history_attention(rows, head)
        o_gpu = got[qs, j * gqa:(j + 1) * gqa].reshape(-1, 128)
        err = P.assert_decode(o_gpu, o_ref, f"prefill 512x32K head {j}")
        e = float(np.abs(gl[qs, j * gqa:(j + 1) * gqa].reshape(-1) - l_ref).max())
        assert e <= 1e-3, f"prefill 512x32K head {j}: lse error {e:.2e}"
        print(f"prefill 512 x 32K head {j}: {len(qs) * gqa} rows, max|o err|={err:.2e} max|lse err|={e:.2e}")
    cache.close()
