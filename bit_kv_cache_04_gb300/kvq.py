"""ctypes binding of libkvq (include/kvq.h), plus a small cache holder.

Argument marshalling only: every step of append, decode attention and
dequantization runs in the library's CUDA kernels.  PyTorch provides device
memory and streams.  Importing this module without a built libkvq.so raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import fields
from typing import Optional, Tuple

from .config import (AXIS_CHANNEL, AXIS_TOKEN, DEV_BOUNDS, DEV_CAPACITY, DEV_LENGTH, DEV_PAGE,  # noqa: F401
                     DEV_RANGE, DEV_STALL, DT_BF16, DT_F16, K_PRE_ROPE, ROTATE_K, ROTATE_V, TBQ4_K, TBQ4_V, ZP_K, ZP_V,
                     Config, Fmt)

_PKG = os.path.dirname(os.path.abspath(__file__))
# KVQ_LIBRARY selects another build of the same ABI (the tests use it for the
# bounds-checked libkvq_checked.so).
LIB_PATH = os.environ.get("KVQ_LIBRARY") or os.path.join(_PKG, "libkvq.so")

STATUS_NAMES = {0: "OK", 1: "ERR_ARG", 2: "ERR_UNSUPPORTED", 3: "ERR_CUDA", 4: "ERR_CAPACITY", 5: "ERR_WORKSPACE"}


class KvqError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class _Fmt(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group", ctypes.c_int32), ("axis", ctypes.c_int32)]


class _Config(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int32), ("H_kv", ctypes.c_int32), ("H_q", ctypes.c_int32), ("D", ctypes.c_int32),
        ("batch", ctypes.c_int32), ("max_T", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
        ("k_fmt", _Fmt), ("v_fmt", _Fmt), ("k_cold", _Fmt), ("v_cold", _Fmt),
        ("hot_window", ctypes.c_int32), ("residual_window", ctypes.c_int32),
        ("flags", ctypes.c_uint32), ("rope_theta", ctypes.c_float), ("sign_seed", ctypes.c_uint64),
        ("page_tokens", ctypes.c_int32), ("n_pages", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class _Cache(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("k_main", "v_main", "k_cold", "v_cold", "k_resid", "v_resid",
                                                  "block_table")]


def _to_c(cfg: Config) -> _Config:
    """kvq_config of a Config."""
    c = _Config()
    for f in fields(cfg):
        v = getattr(cfg, f.name)
        if isinstance(v, Fmt) or (v is None and f.name in ("k_cold", "v_cold")):
            v = v or Fmt(0, 0, 0)
            setattr(c, f.name, _Fmt(v.bits, v.group, v.axis))
        else:
            setattr(c, f.name, v)
    c.reserved = 0
    return c


def _load():
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    vp, i32, i64, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
    cfgp, cachep = P(_Config), P(_Cache)
    sig = {
        "kvq_version": ([], ctypes.c_char_p),
        "kvq_last_error": ([], ctypes.c_char_p),
        "kvq_validate_config": ([cfgp], ctypes.c_int),
        "kvq_block_bytes": ([i32, i32, P(i32)], ctypes.c_int),
        "kvq_bytes_per_token": ([cfgp, P(i64)], ctypes.c_int),
        "kvq_cache_bytes": ([cfgp, i64, P(i64)], ctypes.c_int),
        "kvq_buffer_sizes": ([cfgp, P(sz)], ctypes.c_int),
        "kvq_workspace_bytes": ([cfgp, P(sz)], ctypes.c_int),
        "kvq_workspace_init": ([cfgp, vp, sz, vp], ctypes.c_int),
        "kvq_append": ([cfgp, cachep, i32, i32, vp, vp, vp, vp, i32, i32, vp, sz, vp], ctypes.c_int),
        "kvq_commit_lengths": ([cfgp, vp, vp, vp], ctypes.c_int),
        "kvq_decode_attention": ([cfgp, cachep, i32, i32, vp, vp, vp, i32, vp, sz, vp], ctypes.c_int),
        "kvq_decode_splits": ([cfgp, i32, P(i32)], ctypes.c_int),
        "kvq_decode_step": ([cfgp, cachep, i32, i32, vp, vp, vp, vp, vp, i32, vp, sz, vp], ctypes.c_int),
        "kvq_step_launches": ([cfgp, P(i32)], ctypes.c_int),
        "kvq_launch_counts": ([cfgp, P(i32), P(i32)], ctypes.c_int),
        "kvq_tbq4_codebook": ([P(ctypes.c_float), P(ctypes.c_float)], ctypes.c_int),
        "kvq_decode_attention_static": ([cfgp, cachep, i32, i32, vp, vp, vp, i32, vp], ctypes.c_int),
        "kvq_dequantize": ([cfgp, cachep, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "kvq_test_force_stall": ([i32], ctypes.c_int),
        "kvq_test_shrink_bounds": ([i32], ctypes.c_int),
        "kvq_read_device_status": ([vp, P(u32), vp], ctypes.c_int),
        "kvq_clear_device_status": ([vp, vp], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


LIB = _load()

# C-ABI names declared in include/kvq.h (checked by the tests).
EXPORTED = ("kvq_version", "kvq_last_error", "kvq_validate_config", "kvq_block_bytes", "kvq_bytes_per_token",
            "kvq_cache_bytes", "kvq_buffer_sizes", "kvq_workspace_bytes", "kvq_workspace_init", "kvq_append",
            "kvq_commit_lengths", "kvq_decode_attention", "kvq_decode_splits", "kvq_decode_attention_static",
            "kvq_dequantize", "kvq_launch_counts", "kvq_tbq4_codebook", "kvq_decode_step", "kvq_step_launches",
            "kvq_read_device_status", "kvq_clear_device_status", "kvq_test_force_stall",
            "kvq_test_shrink_bounds")


def _check(st: int):
    if st != 0:
        raise KvqError(st, LIB.kvq_last_error().decode())


# ---- thin wrappers, same names as the C ABI --------------------------------


def kvq_version() -> str:
    return LIB.kvq_version().decode()


def kvq_validate_config(cfg: Config) -> None:
    _check(LIB.kvq_validate_config(ctypes.byref(_to_c(cfg))))


def kvq_block_bytes(bits: int, group: int) -> int:
    out = ctypes.c_int32()
    _check(LIB.kvq_block_bytes(bits, group, ctypes.byref(out)))
    return out.value


def kvq_bytes_per_token(cfg: Config) -> int:
    out = ctypes.c_int64()
    _check(LIB.kvq_bytes_per_token(ctypes.byref(_to_c(cfg)), ctypes.byref(out)))
    return out.value


def kvq_cache_bytes(cfg: Config, T: int) -> int:
    out = ctypes.c_int64()
    _check(LIB.kvq_cache_bytes(ctypes.byref(_to_c(cfg)), T, ctypes.byref(out)))
    return out.value


def kvq_buffer_sizes(cfg: Config) -> Tuple[int, ...]:
    arr = (ctypes.c_size_t * 6)()
    _check(LIB.kvq_buffer_sizes(ctypes.byref(_to_c(cfg)), arr))
    return tuple(arr)


def kvq_tbq4_codebook():
    """(16 centroids, 15 thresholds) of the TBQ4 format, fp32 lists."""
    c = (ctypes.c_float * 16)()
    t = (ctypes.c_float * 15)()
    _check(LIB.kvq_tbq4_codebook(c, t))
    return list(c), list(t)


def kvq_launch_counts(cfg: Config):
    """(kernel launches of one kvq_append call, of one kvq_decode_attention call)."""
    a, d = ctypes.c_int32(), ctypes.c_int32()
    _check(LIB.kvq_launch_counts(ctypes.byref(_to_c(cfg)), ctypes.byref(a), ctypes.byref(d)))
    return a.value, d.value


def kvq_step_launches(cfg: Config) -> int:
    """Kernel launches of one kvq_decode_step call (1 when fused)."""
    n = ctypes.c_int32()
    _check(LIB.kvq_step_launches(ctypes.byref(_to_c(cfg)), ctypes.byref(n)))
    return n.value


def kvq_workspace_bytes(cfg: Config) -> int:
    out = ctypes.c_size_t()
    _check(LIB.kvq_workspace_bytes(ctypes.byref(_to_c(cfg)), ctypes.byref(out)))
    return out.value


def kvq_decode_splits(cfg: Config, n_layers: int) -> int:
    out = ctypes.c_int32()
    _check(LIB.kvq_decode_splits(ctypes.byref(_to_c(cfg)), n_layers, ctypes.byref(out)))
    return out.value


def kvq_test_shrink_bounds(rows: int) -> None:
    """Bounds-checked build: treat the last `rows` rows of every cache segment
    as outside it (0 = off)."""
    _check(LIB.kvq_test_shrink_bounds(rows))


def kvq_test_force_stall(polls: int) -> None:
    """Failure-detection test mode of the tensor-core decode (0 = off)."""
    _check(LIB.kvq_test_force_stall(polls))


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


BUFFER_NAMES = ("k_main", "v_main", "k_cold", "v_cold", "k_resid", "v_resid")


class KVCache:
    """Device buffers (torch tensors) of one quantized cache plus its workspace."""

    def __init__(self, cfg: Config, device="cuda", block_table=None):
        import torch

        self.cfg = cfg
        self.c_cfg = _to_c(cfg)
        self.device = torch.device(device)
        sizes = kvq_buffer_sizes(cfg)
        self.buffers = {}
        for name, n in zip(BUFFER_NAMES, sizes):
            self.buffers[name] = torch.zeros(n, dtype=torch.uint8, device=self.device) if n else None
        self.block_table = None
        if block_table is not None:
            self.block_table = torch.as_tensor(block_table, dtype=torch.int32).to(self.device).contiguous()
        self.ws_bytes = kvq_workspace_bytes(cfg)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.c_cache = _Cache(*[_ptr(self.buffers[n]) for n in BUFFER_NAMES], _ptr(self.block_table))
        _check(LIB.kvq_workspace_init(ctypes.byref(self.c_cfg), _ptr(self.workspace), self.ws_bytes,
                                      _stream(None)))

    # -- the C calls ----------------------------------------------------------

    def append(self, layer0, n_layers, k, v, cu_new, seq_lens, total_new, max_new, stream=None):
        _check(LIB.kvq_append(ctypes.byref(self.c_cfg), ctypes.byref(self.c_cache), layer0, n_layers,
                              _ptr(k), _ptr(v), _ptr(cu_new), _ptr(seq_lens), total_new, max_new,
                              _ptr(self.workspace), self.ws_bytes, _stream(stream)))

    def commit_lengths(self, cu_new, seq_lens, stream=None):
        _check(LIB.kvq_commit_lengths(ctypes.byref(self.c_cfg), _ptr(cu_new), _ptr(seq_lens), _stream(stream)))

    def decode(self, layer0, n_layers, q, seq_lens, out, num_splits=0, stream=None):
        _check(LIB.kvq_decode_attention(ctypes.byref(self.c_cfg), ctypes.byref(self.c_cache), layer0, n_layers,
                                        _ptr(q), _ptr(seq_lens), _ptr(out), num_splits,
                                        _ptr(self.workspace), self.ws_bytes, _stream(stream)))

    def decode_step(self, layer0, n_layers, k_new, v_new, q, seq_lens, out, num_splits=0, stream=None):
        _check(LIB.kvq_decode_step(ctypes.byref(self.c_cfg), ctypes.byref(self.c_cache), layer0, n_layers,
                                   _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(seq_lens), _ptr(out), num_splits,
                                   _ptr(self.workspace), self.ws_bytes, _stream(stream)))

    def dequantize(self, layer, seq, t0, t1, seq_lens, k_out, v_out, stream=None):
        _check(LIB.kvq_dequantize(ctypes.byref(self.c_cfg), ctypes.byref(self.c_cache), layer, seq, t0, t1,
                                  _ptr(seq_lens), _ptr(k_out), _ptr(v_out), _ptr(self.workspace), self.ws_bytes,
                                  _stream(stream)))

    def device_status(self, stream=None) -> int:
        out = ctypes.c_uint32()
        _check(LIB.kvq_read_device_status(_ptr(self.workspace), ctypes.byref(out), _stream(stream)))
        return out.value

    def clear_status(self, stream=None):
        _check(LIB.kvq_clear_device_status(_ptr(self.workspace), _stream(stream)))

    def buffer_numpy(self) -> dict:
        """Host copies of the buffers shaped as the oracle expects (tests only)."""
        import numpy as np

        out = {}
        for n in BUFFER_NAMES:
            t = self.buffers[n]
            if t is not None:
                a = t.cpu().numpy()
                out[n] = a.view(np.uint16) if n.endswith("resid") else a
        return out
