"""C-ABI library: it loads without a GPU, exports every function the header
declares, and validates arguments on the host (no compute calls here)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "oscar.h")


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:oscar_status|const char\*)\s+(oscar_\w+)\s*\(", txt, re.M)))


@pytest.fixture(scope="module")
def O():
    from int2_kv_cache_oscar_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from int2_kv_cache_oscar_gb300 import oscar
    return oscar


def test_header_declares_the_path_calls():
    names = _declared()
    for n in ["oscar_cache_create", "oscar_quantize_append", "oscar_decode_attention",
              "oscar_cache_bytes"]:
        assert n in names


def test_header_is_plain_c(tmp_path):
    """The boundary is a C ABI: the header compiles as strict C99 on its own
    (no C++ or CUDA types leak into the declarations)."""
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    src = tmp_path / "use_header.c"
    src.write_text('#include "oscar.h"\nint main(void) { oscar_cache* c = 0; size_t n = 0;\n'
                   '  return (int)(oscar_cache_bytes(c, -1, 0, &n) == OSCAR_OK); }\n')
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, "-c", str(src),
                        "-o", str(tmp_path / "use_header.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_every_declared_symbol_is_exported(O):
    lib = O.raw_library()
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", O.library_path()], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r" T (oscar_\w+)", out))
    assert set(_declared()) <= exported


@pytest.mark.parametrize("meta_bits,block", [(32, 13824), (0, 13824), (16, 11008)])
def test_required_bytes_layout(O, meta_bits, block):
    cfg = O.make_config(3, 8, 1000, meta_bits=meta_bits)
    n = O.oscar_cache_required_bytes(cfg)
    meta = -(-(256 + 2 * 3 * 8 * 4) // 256) * 256   # status words, value-scale and |value zero| maxima
    groups = -(-1000 // 128)
    blocks = 3 * 8 * groups * block
    win_off = -(-(meta + blocks) // 256) * 256
    assert n == win_off + 3 * 8 * 65536
    # 128 tokens x (32 + 32 code bytes + metadata) per block: 108 or 86 bytes a token
    assert block == 128 * (108 if block == 13824 else 86)


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 64, 4), ("group_size", 64, 4), ("value_group", 16, 4),
    ("max_batch", 0, 1), ("num_kv_heads", 0, 1), ("max_seq_len", 0, 1), ("device", -1, 1),
    ("meta_bits", 8, 4), ("meta_bits", 64, 4)])
def test_bad_configs(O, field, value, status):
    cfg = O.make_config(2, 2, 256)
    setattr(cfg, field, value)
    with pytest.raises(O.OscarError) as e:
        O.oscar_cache_required_bytes(cfg)
    assert e.value.status == status
    assert O.oscar_last_error()


def test_null_arguments_rejected_on_host(O):
    lib = O.raw_library()
    cfg = O.make_config(1, 1, 128)
    h = ctypes.c_void_p(0)
    assert lib.oscar_cache_create(ctypes.byref(cfg), None, 1 << 20, ctypes.byref(h)) == O.OSCAR_ERR_INVALID_ARG
    assert lib.oscar_cache_create(ctypes.byref(cfg), ctypes.c_void_p(256), 10, ctypes.byref(h)) == \
        O.OSCAR_ERR_CAPACITY
    assert lib.oscar_cache_create(ctypes.byref(cfg), ctypes.c_void_p(1000), 1 << 30, ctypes.byref(h)) == \
        O.OSCAR_ERR_INVALID_ARG          # misaligned arena
    assert lib.oscar_quantize_append(None, 1, None, None, None, None, None) == O.OSCAR_ERR_INVALID_ARG
    assert lib.oscar_decode_attention(None, 1, None, None, 4, ctypes.c_float(0), None, None, 0,
                                      None) == O.OSCAR_ERR_INVALID_ARG
    sz = ctypes.c_size_t(0)
    assert lib.oscar_cache_bytes(None, -1, 0, ctypes.byref(sz)) == O.OSCAR_ERR_INVALID_ARG
    assert lib.oscar_cache_destroy(None) == O.OSCAR_OK
    assert lib.oscar_set_timing_events(None, None) == O.OSCAR_OK
    assert lib.oscar_set_timing_events(ctypes.c_void_p(8), None) == O.OSCAR_ERR_INVALID_ARG
    ids = (ctypes.c_int32 * 1)(0)
    lens = (ctypes.c_int32 * 1)(0)
    assert lib.oscar_bf16_decode_attention(1, ids, lens, ctypes.c_void_p(256), ctypes.c_void_p(256), 1,
                                           128, ctypes.c_void_p(256), 4, ctypes.c_float(0),
                                           ctypes.c_void_p(256), ctypes.c_void_p(256), 1 << 20,
                                           None) == O.OSCAR_ERR_INVALID_ARG   # length 0


def test_layout_reader_roundtrip():
    import numpy as np
    from tests import layout
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 4, (128, 128)).astype(np.uint8)
    for order in ("k", "v"):
        words = layout.pack_fragment(codes, order)
        assert np.array_equal(layout.unpack_fragment(words, order), codes)
        # every (row, col) appears exactly once; 16 codes per word
        rows, cols, _ = layout._TABLES[order]
        seen = np.zeros((128, 128), int)
        np.add.at(seen, (rows, cols), 1)
        assert np.all(seen == 1)
    # the two orders hold the same words, permuted: word pair (r = 0, 1) of
    # (mt, j, lane) is 8 contiguous bytes at ((mt*2 + j)*32 + lane)*8 in V order
    wk = layout.pack_fragment(codes, "k").reshape(8, 32, 2, 2)        # [mt][lane][j][r]
    wv = layout.pack_fragment(codes, "v").reshape(8, 2, 32, 2)        # [mt][j][lane][r]
    assert np.array_equal(wk.transpose(0, 2, 1, 3), wv)


def test_layout_reader_fp16_block():
    """The float16-metadata block reader against a block assembled by hand
    from the header's offsets."""
    import numpy as np
    from tests import layout
    rng = np.random.default_rng(6)
    kc = rng.integers(0, 4, (128, 128)).astype(np.uint8)
    vc = rng.integers(0, 4, (128, 128)).astype(np.uint8)
    ks, kz, kn = (rng.standard_normal(128).astype(np.float16) for _ in range(3))
    vs = rng.standard_normal((128, 4)).astype(np.float16)
    vz = rng.standard_normal((128, 4)).astype(np.float16)
    raw = np.zeros(11008, np.uint8)
    raw[0:4096] = layout.pack_fragment(kc).view(np.uint8)
    raw[4096:4352] = ks.view(np.uint8)
    raw[4352:4608] = kz.view(np.uint8)
    raw[4608:4864] = kn.view(np.uint8)
    raw[4864:8960] = layout.pack_fragment(vc.T, "v").view(np.uint8)
    raw[8960:9984] = vs.reshape(-1).view(np.uint8)
    raw[9984:11008] = vz.reshape(-1).view(np.uint8)
    b = layout.parse_block(raw, 16)
    assert np.array_equal(b["kcodes"], kc) and np.array_equal(b["vcodes"], vc)
    assert np.array_equal(b["kscale"], ks.astype(np.float32)) and np.array_equal(b["knorm"], kn.astype(np.float32))
    assert np.array_equal(b["kzero"], kz.astype(np.float32))
    assert np.array_equal(b["vscale"], vs.astype(np.float32)) and np.array_equal(b["vzero"], vz.astype(np.float32))


def test_layout_reader_fp32_block():
    """The float32-metadata block reader against a block assembled by hand
    from the header's offsets."""
    import numpy as np
    from tests import layout
    rng = np.random.default_rng(7)
    kc = rng.integers(0, 4, (128, 128)).astype(np.uint8)
    vc = rng.integers(0, 4, (128, 128)).astype(np.uint8)
    ks, kz, kn = (rng.standard_normal(128).astype(np.float32) for _ in range(3))
    vs = rng.standard_normal((128, 4)).astype(np.float32)
    vz = rng.standard_normal((128, 4)).astype(np.float32)
    raw = np.zeros(13824, np.uint8)
    raw[0:4096] = layout.pack_fragment(kc).view(np.uint8)
    raw[4096:4608] = ks.view(np.uint8)
    raw[4608:5120] = kz.view(np.uint8)
    raw[5120:5632] = kn.view(np.uint8)
    raw[5632:9728] = layout.pack_fragment(vc.T, "v").view(np.uint8)
    rows = [t ^ ((t >> 3) & 1) for t in range(128)]          # header: token t in row t ^ ((t >> 3) & 1)
    vs_st, vz_st = np.empty_like(vs), np.empty_like(vz)
    vs_st[rows], vz_st[rows] = vs, vz
    raw[9728:11776] = vs_st.reshape(-1).view(np.uint8)
    raw[11776:13824] = vz_st.reshape(-1).view(np.uint8)
    b = layout.parse_block(raw)
    assert np.array_equal(b["kcodes"], kc) and np.array_equal(b["vcodes"], vc)
    for name, ref in [("kscale", ks), ("kzero", kz), ("knorm", kn), ("vscale", vs), ("vzero", vz)]:
        assert np.array_equal(b[name], ref), name


def test_binding_checks_buffers_before_any_call():
    """The C ABI sees bare pointers, so the binding checks what it can: dtype,
    contiguity and the shape each call implies.  These raise before the
    library is called (no handle and no GPU needed)."""
    import pytest
    import torch

    from int2_kv_cache_oscar_gb300 import oscar as O

    q = torch.zeros((2, 32, 128), dtype=torch.bfloat16)
    out = torch.zeros_like(q)
    ws = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(ValueError, match="shape"):           # q for 16 heads, 32 requested
        O.oscar_decode_attention(None, [0, 1], q[:, :16].contiguous(), 32, 0.0, out, ws)
    with pytest.raises(ValueError, match="shape"):           # 3 sequences, q for 2
        O.oscar_decode_attention(None, [0, 1, 2], q, 32, 0.0, out, ws)
    with pytest.raises(ValueError, match="contiguous"):
        O.oscar_decode_attention(None, [0, 1], q.transpose(0, 1), 32, 0.0, out, ws)
    with pytest.raises(ValueError, match="bfloat16"):
        O.oscar_decode_attention(None, [0, 1], q.float(), 32, 0.0, out, ws)
    with pytest.raises(TypeError):
        O.oscar_decode_attention(None, [0, 1], [1, 2], 32, 0.0, out, ws)
    k = torch.zeros((10, 8, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="shape"):           # cu_new says 12 rows
        O.oscar_quantize_append(None, [0], [0, 12], k, k)
    with pytest.raises(ValueError, match="shape"):           # v differs from k
        O.oscar_quantize_append(None, [0], [0, 10], k, k[:, :4].contiguous())
    with pytest.raises(ValueError, match="shape"):           # lse for 16 heads
        O.oscar_prefill_attention(None, 0, q, 32, 0.0, out, torch.zeros((2, 16), dtype=torch.float32))
    with pytest.raises(ValueError, match="shape"):           # lse for 1 query row of 2
        O.oscar_prefill_attention(None, 0, q, 32, 0.0, out, torch.zeros((1, 32), dtype=torch.float32))
    with pytest.raises(ValueError, match="shape"):           # k_new for 1 sequence, 2 decoded
        O.oscar_append_decode(None, [0, 1], torch.zeros((1, 8, 128), dtype=torch.bfloat16),
                              torch.zeros((1, 8, 128), dtype=torch.bfloat16), q, 32, 0.0, out, ws)
    with pytest.raises(ValueError, match="first dimension"):  # seq id past the caches
        kc = torch.zeros((1, 8, 256, 128), dtype=torch.bfloat16)
        O.oscar_bf16_decode_attention([0, 1], [10, 10], kc, kc, 8, 256, q, 32, 0.0, out, ws)

