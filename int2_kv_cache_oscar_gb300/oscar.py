"""Thin ctypes binding of liboscar.so (include/oscar.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Device buffers are torch tensors (PyTorch supplies device memory
and streams); host integer arrays are Python sequences.  Every function
raises OscarError when the C call returns a non-zero status.  There is no
CPU fallback: importing this module fails loudly if the library is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liboscar.so")

OSCAR_OK = 0
OSCAR_ERR_INVALID_ARG = 1
OSCAR_ERR_CAPACITY = 2
OSCAR_ERR_CUDA = 3
OSCAR_ERR_UNSUPPORTED = 4
OSCAR_ERR_DEVICE_TIMEOUT = 5

OSCAR_BYTES_USED = 0
OSCAR_BYTES_BF16_EQUIVALENT = 1
OSCAR_BYTES_ARENA = 2

HEAD_DIM = 128
GROUP = 128
VALUE_GROUP = 32
BLOCK_BYTES = 13824
BLOCK_BYTES_META16 = 11008
WINDOW_BYTES = 65536


class OscarError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"oscar status {status}: {message}")
        self.status = status


class oscar_cache_config(ctypes.Structure):
    _fields_ = [("max_batch", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("value_group", ctypes.c_int32),
                ("device", ctypes.c_int32), ("meta_bits", ctypes.c_int32)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"{_LIB_PATH} is missing: build it with int2_kv_cache_oscar_gb300.build.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    I32 = ctypes.c_int32
    SZ = ctypes.c_size_t
    I32P = ctypes.POINTER(ctypes.c_int32)
    sigs = {
        "oscar_cache_required_bytes": [ctypes.POINTER(oscar_cache_config), ctypes.POINTER(SZ)],
        "oscar_cache_create": [ctypes.POINTER(oscar_cache_config), P, SZ, ctypes.POINTER(P)],
        "oscar_cache_destroy": [P],
        "oscar_cache_reset": [P, I32, P],
        "oscar_cache_length": [P, I32, I32P],
        "oscar_quantize_append": [P, I32, I32P, I32P, P, P, P],
        "oscar_decode_workspace_bytes": [P, I32, I32, ctypes.POINTER(SZ)],
        "oscar_decode_attention": [P, I32, I32P, P, I32, ctypes.c_float, P, P, SZ, P],
        "oscar_decode_attention_f32": [P, I32, I32P, P, I32, ctypes.c_float, P, P, SZ, P],
        "oscar_cache_bytes": [P, I32, I32, ctypes.POINTER(SZ)],
        "oscar_cache_block_offset": [P, I32, I32, I32, ctypes.POINTER(SZ)],
        "oscar_cache_window_offset": [P, I32, I32, ctypes.POINTER(SZ)],
        "oscar_cache_check": [P, P],
        "oscar_bf16_decode_workspace_bytes": [I32, I32, I32, ctypes.POINTER(SZ)],
        "oscar_bf16_decode_attention": [I32, I32P, I32P, P, P, I32, I32, P, I32, ctypes.c_float, P, P,
                                        SZ, P],
        "oscar_set_timing_events": [P, P],
        "oscar_test_arm_wait_timeout": [],
        "oscar_test_settled_groups": [P, I32, I32P, P, I32P],
        "oscar_decode_attention_noalloc": [P, I32, I32P, P, I32, ctypes.c_float, P, P],
        "oscar_append_decode": [P, I32, I32P, P, P, P, I32, ctypes.c_float, P, P, SZ, P],
        "oscar_prefill_attention": [P, I32, I32, P, I32, ctypes.c_float, P, P, P, SZ, P],
        "oscar_prefill_workspace_bytes": [P, I32, I32, I32, ctypes.POINTER(SZ)],
    }
    for name, args in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.oscar_last_error.argtypes = []
    lib.oscar_last_error.restype = ctypes.c_char_p
    return lib


_lib = _load()


def library_path() -> str:
    return _LIB_PATH


def raw_library() -> ctypes.CDLL:
    return _lib


def oscar_last_error() -> str:
    return _lib.oscar_last_error().decode()


def _check(status: int):
    if status != OSCAR_OK:
        raise OscarError(status, oscar_last_error())


def _i32(seq: Sequence[int]):
    arr = (ctypes.c_int32 * len(seq))(*[int(x) for x in seq])
    return arr


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _buf(t, dtype, shape, name: str, optional: bool = False) -> ctypes.c_void_p:
    """Pointer of a caller buffer after the checks the C ABI cannot make (it
    receives bare pointers): a torch tensor of `dtype`, dense row-major, whose
    leading dimension is at least shape[0] (the kernels use that many rows) and
    whose other dimensions equal the rest of `shape` (they set the strides);
    None entries are unchecked.  A smaller or differently strided buffer would
    otherwise let a kernel read or write past it."""
    if t is None and optional:
        return ctypes.c_void_p(0)
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None:
        ok = t.dim() == len(shape) and (shape[0] is None or t.shape[0] >= shape[0]) and \
            all(e is None or t.shape[i] == e for i, e in enumerate(shape) if i > 0)
        if not ok:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)} "
                             "(leading dimension at least, None: any)")
    return ctypes.c_void_p(t.data_ptr())


def make_config(max_batch: int, num_kv_heads: int, max_seq_len: int, device: int = 0,
                head_dim: int = HEAD_DIM, group_size: int = GROUP,
                value_group: int = VALUE_GROUP, meta_bits: int = 32) -> oscar_cache_config:
    return oscar_cache_config(max_batch, num_kv_heads, head_dim, max_seq_len, group_size,
                              value_group, device, meta_bits)


def oscar_cache_required_bytes(cfg: oscar_cache_config) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.oscar_cache_required_bytes(ctypes.byref(cfg), ctypes.byref(out)))
    return out.value


def oscar_cache_create(cfg: oscar_cache_config, arena: torch.Tensor) -> ctypes.c_void_p:
    h = ctypes.c_void_p(0)
    _check(_lib.oscar_cache_create(ctypes.byref(cfg), _buf(arena, torch.uint8, None, "arena"),
                                   arena.numel() * arena.element_size(), ctypes.byref(h)))
    return h


def oscar_cache_destroy(handle) -> None:
    _check(_lib.oscar_cache_destroy(handle))


def oscar_cache_reset(handle, seq: int = -1, stream=None) -> None:
    _check(_lib.oscar_cache_reset(handle, seq, _stream(stream)))


def oscar_cache_length(handle, seq: int) -> int:
    out = ctypes.c_int32(0)
    _check(_lib.oscar_cache_length(handle, seq, ctypes.byref(out)))
    return out.value


def oscar_quantize_append(handle, seq_ids: Sequence[int], cu_new: Sequence[int],
                          k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
    rows = int(cu_new[-1]) if len(seq_ids) > 0 else 0
    if rows == 0:
        kp = vp = ctypes.c_void_p(0)
    else:
        kp = _buf(k, torch.bfloat16, (rows, None, HEAD_DIM), "k")
        vp = _buf(v, torch.bfloat16, (rows,) + tuple(k.shape[1:]), "v")
    _check(_lib.oscar_quantize_append(handle, len(seq_ids), _i32(seq_ids), _i32(cu_new), kp, vp,
                                      _stream(stream)))


def oscar_decode_workspace_bytes(handle, n_seqs: int, num_q_heads: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.oscar_decode_workspace_bytes(handle, n_seqs, num_q_heads, ctypes.byref(out)))
    return out.value


def oscar_decode_attention(handle, seq_ids: Sequence[int], q: torch.Tensor, num_q_heads: int,
                           softmax_scale: float, out: torch.Tensor, workspace: torch.Tensor,
                           stream=None) -> None:
    shape = (len(seq_ids), num_q_heads, HEAD_DIM)
    _check(_lib.oscar_decode_attention(handle, len(seq_ids), _i32(seq_ids), _buf(q, torch.bfloat16, shape, "q"),
                                       num_q_heads, ctypes.c_float(softmax_scale),
                                       _buf(out, torch.bfloat16, shape, "out"),
                                       _buf(workspace, torch.uint8, None, "workspace"),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))


def oscar_decode_attention_f32(handle, seq_ids: Sequence[int], q: torch.Tensor, num_q_heads: int,
                               softmax_scale: float, out: torch.Tensor, workspace: torch.Tensor,
                               stream=None) -> None:
    """The same decode with float32 outputs (the merged result before any
    bf16 rounding)."""
    shape = (len(seq_ids), num_q_heads, HEAD_DIM)
    _check(_lib.oscar_decode_attention_f32(handle, len(seq_ids), _i32(seq_ids), _buf(q, torch.bfloat16, shape, "q"),
                                           num_q_heads, ctypes.c_float(softmax_scale),
                                           _buf(out, torch.float32, shape, "out"),
                                           _buf(workspace, torch.uint8, None, "workspace"),
                                           workspace.numel() * workspace.element_size(), _stream(stream)))


def oscar_decode_attention_noalloc(handle, seq_ids: Sequence[int], q: torch.Tensor, num_q_heads: int,
                                   softmax_scale: float, out: torch.Tensor, stream=None) -> None:
    """Decode without a workspace: the partials go to the library's built-in
    device scratch (for callers that cannot allocate device memory)."""
    shape = (len(seq_ids), num_q_heads, HEAD_DIM)
    _check(_lib.oscar_decode_attention_noalloc(handle, len(seq_ids), _i32(seq_ids),
                                               _buf(q, torch.bfloat16, shape, "q"), num_q_heads,
                                               ctypes.c_float(softmax_scale),
                                               _buf(out, torch.bfloat16, shape, "out"), _stream(stream)))


def oscar_append_decode(handle, seq_ids: Sequence[int], k_new: torch.Tensor, v_new: torch.Tensor,
                        q: torch.Tensor, num_q_heads: int, softmax_scale: float, out: torch.Tensor,
                        workspace: torch.Tensor, stream=None) -> None:
    """Append one token per sequence and decode, in one call (one launch when
    no group closes)."""
    shape = (len(seq_ids), num_q_heads, HEAD_DIM)
    kp = _buf(k_new, torch.bfloat16, (len(seq_ids), None, HEAD_DIM), "k_new")
    vp = _buf(v_new, torch.bfloat16, (len(seq_ids),) + tuple(k_new.shape[1:]), "v_new")
    _check(_lib.oscar_append_decode(handle, len(seq_ids), _i32(seq_ids), kp, vp,
                                    _buf(q, torch.bfloat16, shape, "q"), num_q_heads,
                                    ctypes.c_float(softmax_scale), _buf(out, torch.bfloat16, shape, "out"),
                                    _buf(workspace, torch.uint8, None, "workspace"),
                                    workspace.numel() * workspace.element_size(), _stream(stream)))


def oscar_prefill_workspace_bytes(handle, seq: int, n_q: int, num_q_heads: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.oscar_prefill_workspace_bytes(handle, seq, n_q, num_q_heads, ctypes.byref(out)))
    return out.value


def oscar_prefill_attention(handle, seq: int, q: torch.Tensor, num_q_heads: int, softmax_scale: float,
                            out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Attention of a chunk's queries q [n_q, num_q_heads, 128] over the
    sequence's cached tokens; out gets the rows, lse (fp32 [n_q, heads]) their
    log-sum-exp.  With a workspace (uint8, see oscar_prefill_workspace_bytes)
    the history is split across more CTAs and merged."""
    qp = _buf(q, torch.bfloat16, (None, num_q_heads, HEAD_DIM), "q")
    n_q = q.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check(_lib.oscar_prefill_attention(handle, seq, n_q, qp, num_q_heads, ctypes.c_float(softmax_scale),
                                        _buf(out, torch.bfloat16, (n_q, num_q_heads, HEAD_DIM), "out"),
                                        _buf(lse, torch.float32, (n_q, num_q_heads), "lse", optional=True),
                                        _buf(workspace, torch.uint8, (None,), "workspace", optional=True),
                                        ctypes.c_size_t(ws_bytes), _stream(stream)))


def oscar_cache_bytes(handle, seq: int, kind: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.oscar_cache_bytes(handle, seq, kind, ctypes.byref(out)))
    return out.value


def oscar_cache_block_offset(handle, seq: int, kv_head: int, group: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.oscar_cache_block_offset(handle, seq, kv_head, group, ctypes.byref(out)))
    return out.value


def oscar_cache_window_offset(handle, seq: int, kv_head: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.oscar_cache_window_offset(handle, seq, kv_head, ctypes.byref(out)))
    return out.value


def oscar_cache_check(handle, stream=None) -> None:
    _check(_lib.oscar_cache_check(handle, _stream(stream)))


def oscar_bf16_decode_workspace_bytes(n_seqs: int, num_kv_heads: int, num_q_heads: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.oscar_bf16_decode_workspace_bytes(n_seqs, num_kv_heads, num_q_heads,
                                                  ctypes.byref(out)))
    return out.value


def oscar_bf16_decode_attention(seq_ids: Sequence[int], seq_lens: Sequence[int],
                                k_cache: torch.Tensor, v_cache: torch.Tensor, num_kv_heads: int,
                                max_seq_len: int, q: torch.Tensor, num_q_heads: int,
                                softmax_scale: float, out: torch.Tensor, workspace: torch.Tensor,
                                stream=None) -> None:
    cshape = (None, num_kv_heads, max_seq_len, HEAD_DIM)
    if isinstance(k_cache, torch.Tensor) and len(seq_ids) > 0 and k_cache.dim() == 4 and \
            max(int(s) for s in seq_ids) >= k_cache.shape[0]:
        raise ValueError("seq_ids index past the caches' first dimension")
    shape = (len(seq_ids), num_q_heads, HEAD_DIM)
    _check(_lib.oscar_bf16_decode_attention(
        len(seq_ids), _i32(seq_ids), _i32(seq_lens), _buf(k_cache, torch.bfloat16, cshape, "k_cache"),
        _buf(v_cache, torch.bfloat16, cshape, "v_cache"), num_kv_heads, max_seq_len,
        _buf(q, torch.bfloat16, shape, "q"), num_q_heads, ctypes.c_float(softmax_scale),
        _buf(out, torch.bfloat16, shape, "out"), _buf(workspace, torch.uint8, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def oscar_test_arm_wait_timeout() -> None:
    """Test hook: the next INT2 decode on this thread leaves one copy unissued
    so that a bounded device wait runs out (see include/oscar.h)."""
    _check(_lib.oscar_test_arm_wait_timeout())


def oscar_test_settled_groups(cache, seq_ids: Sequence[int], stream=None) -> list:
    """Test hook: per slot, the leading groups the next decode on `stream`
    would copy before its grid dependency wait (see include/oscar.h)."""
    handle = cache.handle if isinstance(cache, OscarCache) else cache
    out = (ctypes.c_int32 * max(len(seq_ids), 1))()
    _check(_lib.oscar_test_settled_groups(handle, len(seq_ids), _i32(seq_ids), _stream(stream), out))
    return [int(out[i]) for i in range(len(seq_ids))]


def oscar_set_timing_events(start: Optional[torch.cuda.Event], stop: Optional[torch.cuda.Event]):
    s = ctypes.c_void_p(0 if start is None else start.cuda_event)
    e = ctypes.c_void_p(0 if stop is None else stop.cuda_event)
    _check(_lib.oscar_set_timing_events(s, e))


class OscarCache:
    """Owns a device arena (a torch uint8 tensor) and the library handle."""

    def __init__(self, max_batch: int, num_kv_heads: int, max_seq_len: int,
                 device: Optional[torch.device] = None, meta_bits: int = 32):
        device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.cfg = make_config(max_batch, num_kv_heads, max_seq_len, device.index or 0, meta_bits=meta_bits)
        self.meta_bits = meta_bits
        nbytes = oscar_cache_required_bytes(self.cfg)
        self.arena = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.handle = oscar_cache_create(self.cfg, self.arena)
        self.num_kv_heads = num_kv_heads
        self.max_batch = max_batch
        self.max_seq_len = max_seq_len

    def close(self):
        if self.handle is not None and self.handle.value:
            oscar_cache_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def length(self, seq: int) -> int:
        return oscar_cache_length(self.handle, seq)

    def append(self, seq_ids, cu_new, k, v, stream=None):
        if isinstance(k, torch.Tensor) and k.dim() == 3 and k.shape[1] != self.num_kv_heads:
            raise ValueError(f"k has {k.shape[1]} KV heads, the cache {self.num_kv_heads}")
        oscar_quantize_append(self.handle, seq_ids, cu_new, k, v, stream)

    def workspace(self, n_seqs: int, num_q_heads: int) -> torch.Tensor:
        n = oscar_decode_workspace_bytes(self.handle, n_seqs, num_q_heads)
        return torch.empty(max(n, 16), dtype=torch.uint8, device=self.arena.device)

    def decode(self, seq_ids, q, num_q_heads, out, workspace, softmax_scale=0.0, stream=None):
        oscar_decode_attention(self.handle, seq_ids, q, num_q_heads, softmax_scale, out, workspace,
                               stream)

    def decode_f32(self, seq_ids, q, num_q_heads, out, workspace, softmax_scale=0.0, stream=None):
        oscar_decode_attention_f32(self.handle, seq_ids, q, num_q_heads, softmax_scale, out, workspace,
                                   stream)

    def append_decode(self, seq_ids, k_new, v_new, q, num_q_heads, out, workspace, softmax_scale=0.0,
                      stream=None):
        if isinstance(k_new, torch.Tensor) and k_new.dim() == 3 and k_new.shape[1] != self.num_kv_heads:
            raise ValueError(f"k_new has {k_new.shape[1]} KV heads, the cache {self.num_kv_heads}")
        oscar_append_decode(self.handle, seq_ids, k_new, v_new, q, num_q_heads, softmax_scale, out, workspace,
                            stream)
