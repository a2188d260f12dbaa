"""CPU-side checks of the C-ABI library: it builds, loads, exports every
symbol include/kvq.h declares, and its host-only logic matches the oracle."""
import os
import re
import subprocess

import numpy as np
import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def kvq():
    from mixed_precision_kv_gb300 import build
    build.build()
    import mixed_precision_kv_gb300 as m
    m.load_library()
    return m


def test_exports_every_declared_symbol(kvq):
    hdr = open(os.path.join(ROOT, "include", "kvq.h")).read()
    declared = set(re.findall(r"KVQ_API\s+[\w\s\*]+?\b(kv_\w+)\s*\(", hdr))
    assert "kv_decode_attn" in declared and len(declared) >= 15
    out = subprocess.run(["nm", "-D", "--defined-only", kvq.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (kv_\w+)", out))
    assert declared <= exported, declared - exported
    assert set(kvq.EXPORTED) == declared
    lib = kvq.load_library()
    for name in declared:
        assert hasattr(lib, name)


def test_alloc_bits_matches_oracle(kvq, orc):
    rng = np.random.default_rng(3)
    for _ in range(300):
        n = int(rng.integers(1, 57))
        N = rng.integers(0, 5000, n)
        D4 = rng.uniform(0.01, 1, n)
        D2 = D4 * (1 + rng.uniform(0.5, 20, n))
        if rng.random() < 0.2:
            D2[: n // 2] = D2[0]          # ties in rho
            D4[: n // 2] = D4[0]
            N[: n // 2] = max(N[0], 1)
        B = (int(rng.integers(0, 5000)), int(rng.integers(1000, 1001)))
        assert np.array_equal(kvq.alloc_bits(N, D2, D4, B), orc.alloc_bits(N, D2, D4, B))


def test_alloc_bits_rejects_bad_budget(kvq):
    with pytest.raises(kvq.KVError) as e:
        kvq.alloc_bits([1, 2], [1.0, 2.0], [0.5, 1.0], (3, 0))
    assert e.value.status == kvq.KV_ERR_INVALID_ARG


def test_workload_bits_agree_between_sides(kvq, orc):
    import kvsynth
    from harness import oracle_bits
    from mixed_precision_kv_gb300.workload import request_bits
    for cfg in (1, 2, 3, 4, 5):
        w = kvsynth.make_workload(cfg, n_req=3, ctx=3000 if cfg != 4 else None)
        for r in range(3):
            assert np.array_equal(request_bits(w, r), oracle_bits(w, r))


def test_alloc_bits3_matches_oracle(kvq, orc):
    rng = np.random.default_rng(31)
    for _ in range(300):
        n = int(rng.integers(1, 57))
        N = rng.integers(0, 300, n).astype(np.int64)
        if rng.integers(0, 4) == 0:
            N[:] = int(rng.integers(1, 40))            # equal counts: many equal savings per bit-token
        D4 = rng.uniform(0.01, 1, n)
        D2 = D4 * (1 + rng.uniform(0.5, 20, n))
        D3 = D4 + (D2 - D4) * rng.uniform(0.0, 1.0, n)
        if rng.integers(0, 4) == 0:
            D3 = (D2 + D4) / 2
        B = (int(rng.integers(18, 42)), 10)
        assert np.array_equal(kvq.alloc_bits3(N, D2, D3, D4, B), orc.alloc_bits3(N, D2, D3, D4, B))
    with pytest.raises(kvq.KVError):
        kvq.alloc_bits3([1, 2], [1.0, 2.0], [0.7, 1.5], [0.5, 1.0], (3, 0))
