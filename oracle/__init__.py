"""CPU oracle for mixed INT2/INT4 paged-KV decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path never
imports this package.  The oracle shares no code with the CUDA path; see
``kvq_oracle.cpp`` for what it computes and which page/section each step
follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.cpp")
_SO = os.path.join(_HERE, "libkvq_oracle.so")
_lock = threading.Lock()
_lib = None

OK, INVALID, OOM, RANGE, STATE = 0, 1, 2, 3, 6
FP4 = 0xF4   # width value of FP4 (E2M1) tokens

_P = ctypes.c_void_p
_I32, _I64, _F32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float


def build(force: bool = False) -> str:
    """Compile the oracle (plain C++17, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fopenmp", "-o", tmp, _SRC])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            sig = {
                "orc_f32_to_f16": (None, [_P, _P, _I64]),
                "orc_f16_to_f32": (None, [_P, _P, _I64]),
                "orc_quant_group": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, _P, _P, _P]),
                "orc_dequant": (_F32, [ctypes.c_uint8, ctypes.c_uint16, ctypes.c_uint16]),
                "orc_alloc_bits": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, _I64, _I64, _P]),
                "orc_alloc_bits3": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int, _I64, _I64, _P]),
                "orc_pool_new": (_P, [ctypes.c_int, _I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, _P,
                                      ctypes.c_int]),
                "orc_fp4_group": (ctypes.c_int, [_P, ctypes.c_int, _P, _P]),
                "orc_e2m1_value": (ctypes.c_double, [ctypes.c_int]),
                "orc_pool_free": (None, [_P]),
                "orc_request_open": (ctypes.c_int, [_P, _P]),
                "orc_request_close": (ctypes.c_int, [_P, _I32]),
                "orc_append": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64]),
                "orc_reorder": (ctypes.c_int, [_P, _P, ctypes.c_int]),
                "orc_evict": (ctypes.c_int, [_P, _P, _P, _I64]),
                "orc_evict_head": (ctypes.c_int, [_P, _P, _P, _P, _I64]),
                "orc_drop_dead_pages": (ctypes.c_int, [_P, _P, ctypes.c_int]),
                "orc_fp_append": (ctypes.c_int, [_P, _I32, _P, _P, _I64]),
                "orc_fp_drop": (ctypes.c_int, [_P, _I32, _I64, _I64]),
                "orc_request_info": (ctypes.c_int, [_P, _I32, _P, _P]),
                "orc_export": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P, _P, _P, _P]),
                "orc_decode": (ctypes.c_int, [_P, _P, _P, ctypes.c_int, ctypes.c_int, _F32, _P, ctypes.c_int,
                                              ctypes.c_int, _P, ctypes.c_int]),
                "orc_num_threads": (ctypes.c_int, []),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


def _check(rc, what):
    if rc != OK:
        raise OracleError(rc, what)


def f32_to_f16(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_f16(_p(x), _p(out), x.size)
    return out


def f16_to_f32(h):
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    lib().orc_f16_to_f32(_p(h), _p(out), h.size)
    return out


def quant_group(x, bits):
    """-> (codes uint8[n], s_bits uint16, z_bits uint16); raises OracleError on range errors."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.empty(x.size, dtype=np.uint8)
    s = np.zeros(1, dtype=np.uint16)
    z = np.zeros(1, dtype=np.uint16)
    _check(lib().orc_quant_group(_p(x), x.size, bits, _p(s), _p(z), _p(codes)), "quant_group")
    return codes, int(s[0]), int(z[0])


def fp4_group(x):
    """FP4 (E2M1) group -> (codes uint8[n], s_bits uint16); raises OracleError on range errors."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.empty(x.size, dtype=np.uint8)
    s = np.zeros(1, dtype=np.uint16)
    _check(lib().orc_fp4_group(_p(x), x.size, _p(s), _p(codes)), "fp4_group")
    return codes, int(s[0])


def e2m1_value(code):
    return float(lib().orc_e2m1_value(int(code)))


def dequant(code, s_bits, z_bits):
    return np.float32(lib().orc_dequant(int(code), int(s_bits), int(z_bits)))


def alloc_bits(N, D2, D4, budget):
    """Greedy INT2/INT4 allocation; budget = (num, den) average bits."""
    N = np.ascontiguousarray(N, dtype=np.int64)
    D2 = np.ascontiguousarray(D2, dtype=np.float64)
    D4 = np.ascontiguousarray(D4, dtype=np.float64)
    out = np.empty(N.size, dtype=np.uint8)
    _check(lib().orc_alloc_bits(_p(N), _p(D2), _p(D4), N.size, int(budget[0]), int(budget[1]), _p(out)),
           "alloc_bits")
    return out


def alloc_bits3(N, D2, D3, D4, budget):
    """Greedy INT2/INT3/INT4 allocation over one-bit steps; budget = (num, den) average bits."""
    N = np.ascontiguousarray(N, dtype=np.int64)
    D2, D3, D4 = (np.ascontiguousarray(d, dtype=np.float64) for d in (D2, D3, D4))
    out = np.empty(N.size, dtype=np.uint8)
    _check(lib().orc_alloc_bits3(_p(N), _p(D2), _p(D3), _p(D4), N.size, int(budget[0]), int(budget[1]), _p(out)),
           "alloc_bits3")
    return out


class OraclePool:
    """Model of the paged pool.  sel_heads: kv heads whose codes are kept;
    n_int3_pages: INT3 page ids [n2 + n4, n2 + n4 + n3), after the INT4 ids;
    n_fp4_pages: FP4 page ids after those."""

    def __init__(self, num_kv_heads, n_int2_pages, n_int4_pages, max_requests, max_pages_per_request,
                 sel_heads=None, n_int3_pages=0, n_fp4_pages=0):
        self.hkv = num_kv_heads
        self.sel = list(range(num_kv_heads)) if sel_heads is None else list(sel_heads)
        sel = np.array(self.sel, dtype=np.int32)
        self.n2 = n_int2_pages
        self.n3 = n_int3_pages
        self.nf = n_fp4_pages
        self.h = lib().orc_pool_new(num_kv_heads, n_int2_pages, n_int3_pages, n_fp4_pages, n_int4_pages,
                                    max_requests, max_pages_per_request, _p(sel), sel.size)
        if not self.h:
            raise OracleError(INVALID, "orc_pool_new")

    def close(self):
        if self.h:
            lib().orc_pool_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def open(self):
        r = np.zeros(1, dtype=np.int32)
        _check(lib().orc_request_open(self.h, _p(r)), "request_open")
        return int(r[0])

    def close_request(self, rid):
        _check(lib().orc_request_close(self.h, rid), "request_close")

    def append(self, req_ids, bits, k=None, v=None):
        """k, v: bf16 bits [n][len(sel)][128] or None (tables only)."""
        req_ids = np.ascontiguousarray(req_ids, dtype=np.int32)
        bits = np.ascontiguousarray(bits, dtype=np.uint8)
        if k is not None:
            k = np.ascontiguousarray(k, dtype=np.uint16)
            v = np.ascontiguousarray(v, dtype=np.uint16)
            assert k.shape == (req_ids.size, len(self.sel), 128)
        return lib().orc_append(self.h, _p(k), _p(v), _p(req_ids), _p(bits), req_ids.size)

    def reorder(self, req_ids):
        req_ids = np.ascontiguousarray(req_ids, dtype=np.int32)
        return lib().orc_reorder(self.h, _p(req_ids), req_ids.size)

    def evict(self, req_ids, pos):
        req_ids = np.ascontiguousarray(req_ids, dtype=np.int32)
        pos = np.ascontiguousarray(pos, dtype=np.int64)
        return lib().orc_evict(self.h, _p(req_ids), _p(pos), req_ids.size)

    def evict_head(self, req_ids, pos, kv_heads):
        """Exclude each (request, position) for one kv head only."""
        req_ids = np.ascontiguousarray(req_ids, dtype=np.int32)
        pos = np.ascontiguousarray(pos, dtype=np.int64)
        kv_heads = np.ascontiguousarray(kv_heads, dtype=np.int32)
        return lib().orc_evict_head(self.h, _p(req_ids), _p(pos), _p(kv_heads), req_ids.size)

    def drop_dead_pages(self, req_ids):
        """Drop every full page with no live slot for any kv head from the listed tables."""
        req_ids = np.ascontiguousarray(req_ids, dtype=np.int32)
        return lib().orc_drop_dead_pages(self.h, _p(req_ids), req_ids.size)

    def fp_append(self, rid, k, v):
        """Full-precision tokens; k, v: bf16 bits [n][len(sel)][128]."""
        k = np.ascontiguousarray(k, dtype=np.uint16)
        v = np.ascontiguousarray(v, dtype=np.uint16)
        assert k.shape == v.shape and k.shape[1:] == (len(self.sel), 128)
        return lib().orc_fp_append(self.h, rid, _p(k), _p(v), k.shape[0])

    def fp_drop(self, rid, first, n):
        return lib().orc_fp_drop(self.h, rid, first, n)

    def info(self, rid):
        n_pages = np.zeros(1, dtype=np.int32)
        n_tok = np.zeros(1, dtype=np.int64)
        _check(lib().orc_request_info(self.h, rid, _p(n_pages), _p(n_tok)), "request_info")
        return int(n_pages[0]), int(n_tok[0])

    def export(self, rid, content=True):
        n, _ = self.info(rid)
        ns = len(self.sel)
        d = dict(ids=np.zeros(n, np.int32), is_int2=np.zeros(n, np.uint8), fill=np.zeros(n, np.uint8),
                 live=np.zeros(n, np.uint32))
        if content:
            d.update(kc=np.zeros((n, ns, 32, 128), np.uint8), vc=np.zeros((n, ns, 32, 128), np.uint8),
                     km=np.zeros((n, ns, 256), np.uint16), vm=np.zeros((n, ns, 256), np.uint16))
        _check(lib().orc_export(self.h, rid, _p(d["ids"]), _p(d["is_int2"]), _p(d["fill"]), _p(d["live"]),
                                _p(d.get("kc")), _p(d.get("vc")), _p(d.get("km")), _p(d.get("vm"))), "export")
        return d

    def decode(self, q_bits, req_ids, softmax_scale, pairs=None, n_splits=1, n_threads=0):
        """q_bits: bf16 bits [B][Hq][128].  Returns fp64 [n_pairs][128] (all pairs if None)."""
        q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
        B, Hq, _ = q_bits.shape
        req_ids = np.ascontiguousarray(req_ids, dtype=np.int32)
        if pairs is None:
            pairs = np.array([(b, h) for b in range(B) for h in range(Hq)], dtype=np.int32)
        pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        out = np.zeros((pairs.shape[0], 128), dtype=np.float64)
        _check(lib().orc_decode(self.h, _p(q_bits), _p(req_ids), B, Hq, float(softmax_scale), _p(pairs),
                                pairs.shape[0], n_splits, _p(out), n_threads), "decode")
        return out


def num_threads():
    return int(lib().orc_num_threads())
