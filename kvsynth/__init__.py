"""Seeded synthetic inputs for the mixed INT2/INT4 paged-KV decode path.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests.  It holds none of the KV-cache method's arithmetic: it draws tags,
distortion tables, context lengths, eviction sets and bf16 tensors, nothing
else.  Element values come from a counter-based generator (Philox4x32-10 +
Irwin-Hall(12), see ``csrc/kvsynth_gen.h``) that has one host and one device
implementation producing identical bits, so the oracle can regenerate any
sampled row that the GPU path generated on the device.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_CSRC = os.path.join(_HERE, "csrc")
_HOST_SO = os.path.join(_HERE, "libkvsynth_host.so")
_DEV_SO = os.path.join(_HERE, "libkvsynth_dev.so")
_lock = threading.Lock()
_host = None
_dev = None

TENSOR_K, TENSOR_V, TENSOR_Q = 1, 2, 3


def build_host(force: bool = False) -> str:
    src = os.path.join(_CSRC, "kvsynth_host.c")
    if force or not os.path.exists(_HOST_SO) or os.path.getmtime(_HOST_SO) < max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(_CSRC, "kvsynth_gen.h"))):
        tmp = _HOST_SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, src])
        os.replace(tmp, _HOST_SO)
    return _HOST_SO


def build_dev(force: bool = False) -> str:
    src = os.path.join(_CSRC, "kvsynth_dev.cu")
    if force or not os.path.exists(_DEV_SO) or os.path.getmtime(_DEV_SO) < max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(_CSRC, "kvsynth_gen.h"))):
        tmp = _DEV_SO + f".tmp{os.getpid()}"
        subprocess.check_call(["nvcc", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-Xcompiler", "-fPIC", "-shared", "--fmad=false", "-o", tmp, src])
        os.replace(tmp, _DEV_SO)
    return _DEV_SO


def _host_lib():
    global _host
    with _lock:
        if _host is None:
            lib = ctypes.CDLL(build_host())
            lib.kvs_fill_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int64,
                                          ctypes.c_void_p, ctypes.c_void_p]
            lib.kvs_fill_bf16.restype = None
            lib.kvs_fill_bf16_heads.argtypes = lib.kvs_fill_bf16.argtypes + [ctypes.c_void_p, ctypes.c_int32]
            lib.kvs_fill_bf16_heads.restype = None
            lib.kvs_philox_blocks.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            lib.kvs_philox_blocks.restype = None
            _host = lib
    return _host


def _dev_lib():
    global _dev
    with _lock:
        if _dev is None:
            if not os.path.exists(_DEV_SO):
                raise RuntimeError("libkvsynth_dev.so is not built; run __graft_entry__.build()")
            lib = ctypes.CDLL(_DEV_SO)
            lib.kvs_fill_bf16_dev.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int64,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            lib.kvs_fill_bf16_dev.restype = ctypes.c_int
            _dev = lib
    return _dev


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def fill_bf16_host(n_tok, H, D, seed, tensor, stream, tok0=0, chan_mult=None, row_mult=None):
    """bf16 bits, shape [n_tok][H][D], generated on the host."""
    out = np.empty((n_tok, H, D), dtype=np.uint16)
    cm = None if chan_mult is None else np.ascontiguousarray(chan_mult, dtype=np.float32)
    rm = None if row_mult is None else np.ascontiguousarray(row_mult, dtype=np.float32)
    _host_lib().kvs_fill_bf16(_ptr(out), n_tok, H, D, seed, tensor, stream, tok0, _ptr(cm), _ptr(rm))
    return out


def fill_bf16_host_heads(n_tok, H, D, seed, tensor, stream, heads, tok0=0, chan_mult=None, row_mult=None):
    """Like fill_bf16_host but only for the listed heads: shape [n_tok][len(heads)][D]."""
    heads = np.ascontiguousarray(heads, dtype=np.int32)
    out = np.empty((n_tok, heads.size, D), dtype=np.uint16)
    cm = None if chan_mult is None else np.ascontiguousarray(chan_mult, dtype=np.float32)
    rm = None if row_mult is None else np.ascontiguousarray(row_mult, dtype=np.float32)
    _host_lib().kvs_fill_bf16_heads(_ptr(out), n_tok, H, D, seed, tensor, stream, tok0, _ptr(cm), _ptr(rm),
                                    _ptr(heads), heads.size)
    return out


def fill_bf16_dev(out_ptr, n_tok, H, D, seed, tensor, stream, tok0=0, chan_mult_ptr=None,
                  row_mult_ptr=None, cuda_stream=0):
    """Same values as fill_bf16_host, written by a device kernel to out_ptr."""
    rc = _dev_lib().kvs_fill_bf16_dev(ctypes.c_void_p(out_ptr), n_tok, H, D, seed, tensor, stream, tok0,
                                      ctypes.c_void_p(chan_mult_ptr or 0), ctypes.c_void_p(row_mult_ptr or 0),
                                      ctypes.c_void_p(cuda_stream or 0))
    if rc != 0:
        raise RuntimeError(f"kvs_fill_bf16_dev failed with CUDA error {rc}")


def philox_blocks_host(ctr: np.ndarray, key: np.ndarray) -> np.ndarray:
    ctr = np.ascontiguousarray(ctr, dtype=np.uint32).reshape(-1, 4)
    key = np.ascontiguousarray(key, dtype=np.uint32).reshape(-1, 2)
    out = np.empty_like(ctr)
    _host_lib().kvs_philox_blocks(_ptr(ctr), _ptr(key), _ptr(out), ctr.shape[0])
    return out


def philox_blocks_np(ctr: np.ndarray, key: np.ndarray) -> np.ndarray:
    """Plain numpy Philox4x32-10 (Salmon et al., SC'11) for cross-checking the C version."""
    c = np.array(ctr, dtype=np.uint64).reshape(-1, 4).copy()
    k = np.array(key, dtype=np.uint64).reshape(-1, 2).copy()
    m = np.uint64(0xFFFFFFFF)
    for r in range(10):
        if r > 0:
            k[:, 0] = (k[:, 0] + np.uint64(0x9E3779B9)) & m
            k[:, 1] = (k[:, 1] + np.uint64(0xBB67AE85)) & m
        p0 = np.uint64(0xD2511F53) * c[:, 0]
        p1 = np.uint64(0xCD9E8D57) * c[:, 2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & m
        hi1, lo1 = p1 >> np.uint64(32), p1 & m
        c = np.stack([hi1 ^ c[:, 1] ^ k[:, 0], lo1, hi0 ^ c[:, 3] ^ k[:, 1], lo0], axis=1)
    return c.astype(np.uint32)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


from .recipes import Workload, RequestSpec, make_workload, tag_runs  # noqa: E402,F401
