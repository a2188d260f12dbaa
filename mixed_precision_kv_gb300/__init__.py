"""Mixed INT2/INT4 paged KV cache with fused-dequant split-KV decode attention
for GB300 (sm_103a).

This package is a thin ctypes binding over ``libkvq.so`` (C ABI declared in
``include/kvq.h``).  It only marshals arguments: every step of the path runs
in the library's CUDA kernels.  PyTorch supplies device memory and streams.
There is no CPU fallback: if the library is missing, importing
``mixed_precision_kv_gb300`` works but creating a pool raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_OOM, KV_ERR_RANGE, KV_ERR_CUDA, KV_ERR_DEVICE_TIMEOUT, KV_ERR_STATE = range(7)
KV_DECODE_AUTO, KV_DECODE_SIMT, KV_DECODE_MMA = 0, 1, 2
HEAD_DIM, PAGE_TOKENS, GROUP = 128, 32, 32
KV_WIDTH_FP4 = 0xF4   # width value of FP4 (E2M1) tokens

EXPORTED = ["kv_pool_create", "kv_pool_destroy", "kv_request_open", "kv_request_close", "kv_append_quant",
            "kv_reorder_pages", "kv_evict_slots", "kv_decode_attn", "kv_set_decode_impl", "kv_pool_sync",
            "kv_request_info", "kv_export_request", "kv_last_decode_stats", "kv_pool_launch_count", "kv_alloc_bits",
            "kv_last_error", "kv_decode_attn_noalloc", "kv_decode_timing", "kv_evict_slots_head", "kv_fp_configure",
            "kv_fp_append", "kv_fp_drop", "kv_fp_count", "kv_set_wait_limit", "kv_drop_dead_pages",
            "kv_decode_attn_groups", "kv_alloc_bits3"]

_P = ctypes.c_void_p
_I32, _I64 = ctypes.c_int32, ctypes.c_int64
_lock = threading.Lock()
_lib = None


class KVConfig(ctypes.Structure):
    _fields_ = [("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("page_tokens", ctypes.c_int32),
                ("group", ctypes.c_int32), ("n_int2_pages", ctypes.c_int64), ("n_int4_pages", ctypes.c_int64),
                ("max_requests", ctypes.c_int32), ("max_pages_per_request", ctypes.c_int32),
                ("device", ctypes.c_int32), ("n_int3_pages", ctypes.c_int64), ("n_fp4_pages", ctypes.c_int64)]


class KVError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"[kv status {status}] {msg}")
        self.status = status


def load_library(path: str = LIB_PATH):
    """Load libkvq.so and declare its signatures (raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        sig = {
            "kv_pool_create": [ctypes.POINTER(KVConfig), ctypes.POINTER(_P)],
            "kv_pool_destroy": [_P],
            "kv_request_open": [_P, _P],
            "kv_request_close": [_P, _I32],
            "kv_append_quant": [_P, _P, _P, _P, _P, _I64, _P],
            "kv_reorder_pages": [_P, _P, _I32, _P],
            "kv_evict_slots": [_P, _P, _P, _I64, _P],
            "kv_evict_slots_head": [_P, _P, _P, _P, _I64, _P],
            "kv_drop_dead_pages": [_P, _P, _I32, _P],
            "kv_decode_attn_groups": [_P, _I32, _P, _P, _I32, _I32, ctypes.c_float, _P, _P],
            "kv_fp_configure": [_P, _I32],
            "kv_fp_append": [_P, _P, _P, _P, _I64, _P],
            "kv_fp_drop": [_P, _I32, _I64, _I64, _P],
            "kv_fp_count": [_P, _I32, _P],
            "kv_decode_attn": [_P, _P, _P, _I32, _I32, ctypes.c_float, _P, _P],
            "kv_decode_attn_noalloc": [_P, _P, _P, _I32, _I32, ctypes.c_float, _P, _P],
            "kv_set_decode_impl": [_P, _I32],
            "kv_set_wait_limit": [_P, _I64],
            "kv_pool_sync": [_P],
            "kv_request_info": [_P, _I32, _P, _P],
            "kv_export_request": [_P, _I32, _P, _P, _P, _P, _P, _P, _P, _P],
            "kv_last_decode_stats": [_P, _P, _P, _P],
            "kv_pool_launch_count": [_P, _P],
            "kv_decode_timing": [_P, _I32, _P, _P, _P],
            "kv_alloc_bits": [_P, _P, _P, _I32, _I64, _I64, _P],
            "kv_alloc_bits3": [_P, _P, _P, _P, _I32, _I64, _I64, _P],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.kv_last_error.argtypes = []
        L.kv_last_error.restype = ctypes.c_char_p
        _lib = L
        return L


def _check(rc, what):
    if rc != KV_OK:
        msg = load_library().kv_last_error().decode(errors="replace")
        raise KVError(rc, f"{what}: {msg}")


def _np(a, dtype):
    if type(a) is np.ndarray and a.dtype == dtype and a.flags.c_contiguous:
        return a
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data


_torch = None
_raw_stream = None


def _torch_mod():
    global _torch, _raw_stream
    if _torch is None:
        import torch
        _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _torch = torch
    return _torch


def _stream(stream, device):
    """cudaStream_t (as an int) of `stream`, or of torch's current stream on `device`."""
    if stream is not None:
        return stream.cuda_stream
    torch = _torch_mod()
    if _raw_stream is not None:
        return _raw_stream(device)
    return torch.cuda.current_stream(device).cuda_stream


def alloc_bits(N, D2, D4, budget):
    """Greedy INT2/INT4 bit allocation (host); budget = (num, den) average bits."""
    N = _np(N, np.int64)
    D2 = _np(D2, np.float64)
    D4 = _np(D4, np.float64)
    out = np.empty(N.size, dtype=np.uint8)
    _check(load_library().kv_alloc_bits(_ptr(N), _ptr(D2), _ptr(D4), N.size, int(budget[0]), int(budget[1]),
                                        _ptr(out)), "kv_alloc_bits")
    return out


def alloc_bits3(N, D2, D3, D4, budget):
    """Greedy INT2/INT3/INT4 bit allocation over one-bit steps (host); budget = (num, den)."""
    N = _np(N, np.int64)
    D2, D3, D4 = _np(D2, np.float64), _np(D3, np.float64), _np(D4, np.float64)
    out = np.empty(N.size, dtype=np.uint8)
    _check(load_library().kv_alloc_bits3(_ptr(N), _ptr(D2), _ptr(D3), _ptr(D4), N.size, int(budget[0]),
                                         int(budget[1]), _ptr(out)), "kv_alloc_bits3")
    return out


class KVPool:
    """A paged INT2/INT4 pool on one GPU (see include/kvq.h for every call's contract)."""

    def __init__(self, num_kv_heads, n_int2_pages, n_int4_pages, max_requests, max_pages_per_request, device=0,
                 n_int3_pages=0, n_fp4_pages=0):
        L = load_library()
        cfg = KVConfig(num_kv_heads, HEAD_DIM, PAGE_TOKENS, GROUP, n_int2_pages, n_int4_pages, max_requests,
                       max_pages_per_request, device, n_int3_pages, n_fp4_pages)
        h = _P()
        _check(L.kv_pool_create(ctypes.byref(cfg), ctypes.byref(h)), "kv_pool_create")
        self._h = h
        self._L = L
        self.num_kv_heads = num_kv_heads
        self.n_int2_pages = n_int2_pages
        self.n_int3_pages = n_int3_pages
        self.n_fp4_pages = n_fp4_pages
        self.device = device

    @property
    def handle(self):
        return self._h

    def destroy(self):
        if getattr(self, "_h", None):
            load_library().kv_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    def open(self) -> int:
        r = ctypes.c_int32()
        _check(load_library().kv_request_open(self._h, ctypes.byref(r)), "kv_request_open")
        return r.value

    def close_request(self, rid):
        _check(load_library().kv_request_close(self._h, int(rid)), "kv_request_close")

    def append(self, k, v, req_ids, bits, stream=None):
        """k, v: torch bf16 CUDA tensors [n][Hkv][128]; req_ids, bits: host sequences [n]."""
        req_ids = _np(req_ids, np.int32)
        bits = _np(bits, np.uint8)
        n = req_ids.size
        if bits.size != n:
            raise ValueError("bits and req_ids differ in length")
        if n:
            self._check_kv(k, n)
            self._check_kv(v, n)
        rc = self._L.kv_append_quant(self._h, k.data_ptr() if n else None, v.data_ptr() if n else None,
                                     req_ids.ctypes.data, bits.ctypes.data, n, _stream(stream, self.device))
        if rc:
            _check(rc, "kv_append_quant")

    def _check_kv(self, t, n):
        torch = _torch_mod()
        if t.dtype is not torch.bfloat16 or not self._on_pool_device(t) or \
                t.shape != (n, self.num_kv_heads, HEAD_DIM) or not t.is_contiguous():
            raise ValueError(f"expected a contiguous bf16 tensor [{n}][{self.num_kv_heads}][128] on the pool's "
                             f"device")

    def reorder(self, req_ids, stream=None):
        req_ids = _np(req_ids, np.int32)
        rc = self._L.kv_reorder_pages(self._h, req_ids.ctypes.data, req_ids.size, _stream(stream, self.device))
        if rc:
            _check(rc, "kv_reorder_pages")

    def evict(self, req_ids, token_pos, stream=None):
        req_ids = _np(req_ids, np.int32)
        token_pos = _np(token_pos, np.int64)
        if req_ids.size != token_pos.size:
            raise ValueError("req_ids and token_pos differ in length")
        _check(load_library().kv_evict_slots(self._h, _ptr(req_ids), _ptr(token_pos), req_ids.size,
                                             _stream(stream, self.device)), "kv_evict_slots")

    def evict_head(self, req_ids, token_pos, kv_heads, stream=None):
        """kv_evict_slots_head: each (request, position) reads as dead for one kv head."""
        req_ids = _np(req_ids, np.int32)
        token_pos = _np(token_pos, np.int64)
        kv_heads = _np(kv_heads, np.int32)
        if not (req_ids.size == token_pos.size == kv_heads.size):
            raise ValueError("req_ids, token_pos and kv_heads differ in length")
        _check(load_library().kv_evict_slots_head(self._h, _ptr(req_ids), _ptr(token_pos), _ptr(kv_heads),
                                                  req_ids.size, _stream(stream, self.device)), "kv_evict_slots_head")

    def drop_dead_pages(self, req_ids, stream=None):
        """kv_drop_dead_pages: free every full page with no live slot for any kv head."""
        req_ids = _np(req_ids, np.int32)
        _check(load_library().kv_drop_dead_pages(self._h, _ptr(req_ids), req_ids.size, _stream(stream, self.device)),
               "kv_drop_dead_pages")

    def fp_configure(self, max_tokens):
        """kv_fp_configure: capacity of every request's full-precision lists."""
        _check(load_library().kv_fp_configure(self._h, int(max_tokens)), "kv_fp_configure")

    def fp_append(self, req_ids, k, v, stream=None):
        """kv_fp_append: k, v torch bf16 CUDA tensors [n][Hkv][128]; req_ids: a request id
        (every token) or a host sequence [n]."""
        n = int(k.shape[0])
        req_ids = np.full(n, int(req_ids), np.int32) if np.ndim(req_ids) == 0 else _np(req_ids, np.int32)
        if req_ids.size != n:
            raise ValueError("req_ids and k differ in length")
        if n:
            self._check_kv(k, n)
            self._check_kv(v, n)
        _check(load_library().kv_fp_append(self._h, k.data_ptr() if n else None, v.data_ptr() if n else None,
                                           _ptr(req_ids), n, _stream(stream, self.device)), "kv_fp_append")

    def fp_drop(self, rid, first, n, stream=None):
        _check(load_library().kv_fp_drop(self._h, int(rid), int(first), int(n), _stream(stream, self.device)),
               "kv_fp_drop")

    def fp_count(self, rid) -> int:
        n = ctypes.c_int64(0)
        _check(load_library().kv_fp_count(self._h, int(rid), ctypes.byref(n)), "kv_fp_count")
        return int(n.value)

    def _on_pool_device(self, t):
        return t.is_cuda and t.device.index == self.device

    def decode(self, q, req_ids, softmax_scale, out=None, stream=None):
        """q: torch bf16 CUDA [B][Hq][128] -> out fp32 [B][Hq][128], both on the pool's device."""
        torch = _torch_mod()
        req_ids = _np(req_ids, np.int32)
        B, Hq, D = q.shape
        if q.dtype is not torch.bfloat16 or not self._on_pool_device(q) or D != HEAD_DIM or B != req_ids.size or \
                not q.is_contiguous():
            raise ValueError("q must be a contiguous bf16 tensor [B][Hq][128] on the pool's device with "
                             "B == len(req_ids)")
        if out is None:
            out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
        elif out.dtype is not torch.float32 or out.shape != q.shape or not self._on_pool_device(out) or \
                not out.is_contiguous():
            raise ValueError("out must be a contiguous fp32 tensor shaped like q on the pool's device")
        rc = self._L.kv_decode_attn(self._h, q.data_ptr(), req_ids.ctypes.data, B, Hq, softmax_scale,
                                    out.data_ptr(), _stream(stream, self.device))
        if rc:
            _check(rc, "kv_decode_attn")
        return out

    def decode_noalloc(self, q, req_ids, softmax_scale, out, stream=None):
        """kv_decode_attn_noalloc: like decode(), but the library allocates no device
        memory (fixed internal scratch); the caller passes a preallocated `out`.
        Issue it on the stream that carries the pool's other work."""
        torch = _torch_mod()
        req_ids = _np(req_ids, np.int32)
        B, Hq, D = q.shape
        if q.dtype is not torch.bfloat16 or not self._on_pool_device(q) or not q.is_contiguous() or \
                D != HEAD_DIM or B != req_ids.size:
            raise ValueError("q must be a contiguous bf16 tensor [B][Hq][128] on the pool's device with "
                             "B == len(req_ids)")
        if out.dtype is not torch.float32 or not self._on_pool_device(out) or not out.is_contiguous() or \
                tuple(out.shape) != (B, Hq, D):
            raise ValueError("out must be a contiguous fp32 tensor shaped like q on the pool's device")
        _check(load_library().kv_decode_attn_noalloc(self._h, ctypes.c_void_p(q.data_ptr()), _ptr(req_ids), B, Hq,
                                                     float(softmax_scale), ctypes.c_void_p(out.data_ptr()),
                                                     _stream(stream, self.device)), "kv_decode_attn_noalloc")
        return out

    @staticmethod
    def decode_groups(pools, q, req_ids, softmax_scale, out=None, stream=None):
        """kv_decode_attn_groups: pools hold consecutive kv head ranges of one model
        (pools[0]'s first); req_ids [n_pools][B]: each pool's request of batch row b.
        q: torch bf16 CUDA [B][Hq][128] -> out fp32 [B][Hq][128]."""
        torch = _torch_mod()
        pools = list(pools)
        if not pools:
            raise ValueError("need at least one pool")
        req_ids = _np(req_ids, np.int32)
        B, Hq, D = q.shape
        dev = pools[0].device
        if req_ids.shape != (len(pools), B):
            raise ValueError("req_ids must be [n_pools][B]")
        if q.dtype is not torch.bfloat16 or not pools[0]._on_pool_device(q) or D != HEAD_DIM or \
                not q.is_contiguous():
            raise ValueError("q must be a contiguous bf16 tensor [B][Hq][128] on the pools' device")
        if out is None:
            out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
        elif out.dtype is not torch.float32 or out.shape != q.shape or not pools[0]._on_pool_device(out) or \
                not out.is_contiguous():
            raise ValueError("out must be a contiguous fp32 tensor shaped like q on the pools' device")
        handles = (_P * len(pools))(*[p._h for p in pools])
        _check(load_library().kv_decode_attn_groups(handles, len(pools), ctypes.c_void_p(q.data_ptr()),
                                                    _ptr(req_ids), B, Hq, float(softmax_scale),
                                                    ctypes.c_void_p(out.data_ptr()), _stream(stream, dev)),
               "kv_decode_attn_groups")
        return out

    def set_wait_limit(self, first_wait_spins):
        """kv_set_wait_limit: bound of the scans' first copy wait (testing the timeout
        path); -1 restores the normal bound."""
        _check(load_library().kv_set_wait_limit(self._h, int(first_wait_spins)), "kv_set_wait_limit")

    def set_decode_impl(self, impl):
        _check(load_library().kv_set_decode_impl(self._h, int(impl)), "kv_set_decode_impl")

    def sync(self):
        _check(load_library().kv_pool_sync(self._h), "kv_pool_sync")

    def info(self, rid):
        n_pages = ctypes.c_int32()
        n_tok = ctypes.c_int64()
        _check(load_library().kv_request_info(self._h, int(rid), ctypes.byref(n_pages), ctypes.byref(n_tok)),
               "kv_request_info")
        return n_pages.value, n_tok.value

    def export(self, rid, content=True):
        n, _ = self.info(rid)
        H = self.num_kv_heads
        d = dict(ids=np.zeros(n, np.int32), is_int2=np.zeros(n, np.uint8), fill=np.zeros(n, np.uint8),
                 live=np.zeros(n, np.uint32))
        if content:
            d.update(kc=np.zeros((n, H, 32, 128), np.uint8), vc=np.zeros((n, H, 32, 128), np.uint8),
                     km=np.zeros((n, H, 256), np.uint16), vm=np.zeros((n, H, 256), np.uint16))
        _check(load_library().kv_export_request(self._h, int(rid), _ptr(d["ids"]), _ptr(d["is_int2"]),
                                                _ptr(d["fill"]), _ptr(d["live"]), _ptr(d.get("kc")),
                                                _ptr(d.get("vc")), _ptr(d.get("km")), _ptr(d.get("vm"))),
               "kv_export_request")
        return d

    def decode_timing(self, enable=True, every=1):
        """(Re)start (recording every `every`-th decode call) or stop device timing
        of the decode kernels; returns (n_calls, mean scan ms, mean scan+merge ms)
        recorded since the last start."""
        n = ctypes.c_int64()
        a = ctypes.c_float()
        b = ctypes.c_float()
        _check(load_library().kv_decode_timing(self._h, int(every) if enable else 0, ctypes.byref(n),
                                               ctypes.byref(a), ctypes.byref(b)), "kv_decode_timing")
        return n.value, a.value, b.value

    def launch_count(self) -> int:
        n = ctypes.c_int64()
        _check(load_library().kv_pool_launch_count(self._h, ctypes.byref(n)), "kv_pool_launch_count")
        return n.value

    def last_decode_stats(self):
        b = ctypes.c_int64()
        s = ctypes.c_int32()
        p = ctypes.c_int64()
        _check(load_library().kv_last_decode_stats(self._h, ctypes.byref(b), ctypes.byref(s), ctypes.byref(p)),
               "kv_last_decode_stats")
        return dict(kv_bytes=b.value, n_splits=s.value, n_pages=p.value)
