"""The C ABI from a plain C11 program (tests/c_abi/kvq_c_client.c), without the
Python binding: it compiles and links against include/kvq.h and libkvq.so
alone (CPU), and on the GPU its decode output matches the oracle's fp64
attention on the same inputs."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import kvsynth
import oracle
from harness import assert_outputs_close

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "kvq_c_client.c")
LIBDIR = os.path.join(ROOT, "mixed_precision_kv_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    """The client built against the in-tree library (rpath set to it)."""
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA runtime headers are not available")
    from mixed_precision_kv_gb300 import build as kbuild
    kbuild.build()
    exe = str(tmp_path_factory.mktemp("c_abi") / "kvq_c_client")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-O2",
           "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(CUDA, "include"), SRC,
           "-L" + LIBDIR, "-lkvq", "-L" + os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath-link," + os.path.join(CUDA, "lib64"), "-Wl,-rpath," + LIBDIR, "-o", exe]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    assert r.returncode == 0, r.stdout
    return exe


def test_c_client_compiles_and_links(client):
    assert os.access(client, os.X_OK)


@pytest.mark.gpu
def test_c_client_matches_oracle(client, tmp_path):
    """Three requests (1500, 700 and 97 tokens, mixed widths) appended in one
    call each, 40 evictions, reorder, decode at g = 4: outputs within max-abs
    1e-3 / relative-L2 1e-4 of the oracle, token counts as appended."""
    hkv, hq, seed = 2, 8, 777
    lens = [1500, 700, 97]
    rng = np.random.default_rng(5)
    bits = [np.where(rng.random(n) < p, 2, 4).astype(np.uint8) for n, p in zip(lens, [0.6, 0.3, 0.8])]
    ks = [kvsynth.fill_bf16_host(n, hkv, 128, seed, kvsynth.TENSOR_K, r) for r, n in enumerate(lens)]
    vs = [kvsynth.fill_bf16_host(n, hkv, 128, seed, kvsynth.TENSOR_V, r) for r, n in enumerate(lens)]
    ev_req = np.concatenate([np.full(20, 0), np.full(20, 1)]).astype(np.int32)
    ev_pos = np.concatenate([rng.choice(lens[0], 20, replace=False),
                             rng.choice(lens[1], 20, replace=False)]).astype(np.int64)
    q = kvsynth.fill_bf16_host(len(lens), hq, 128, seed, kvsynth.TENSOR_Q, 0)
    scale = np.float32(1 / np.sqrt(128))
    inp = tmp_path / "in.bin"
    with open(inp, "wb") as f:
        f.write(np.array([hkv, hq, len(lens)], np.int32).tobytes())
        f.write(np.array(lens, np.int32).tobytes())
        f.write(np.array([scale], np.float32).tobytes())
        for b, k, v in zip(bits, ks, vs):
            f.write(b.tobytes())
            f.write(np.ascontiguousarray(k).tobytes())
            f.write(np.ascontiguousarray(v).tobytes())
        f.write(np.array([ev_req.size], np.int64).tobytes())
        f.write(ev_req.tobytes())
        f.write(ev_pos.tobytes())
        f.write(np.ascontiguousarray(q).tobytes())
    outp = tmp_path / "out.bin"
    r = subprocess.run([client, str(inp), str(outp)], stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout
    raw = np.fromfile(outp, dtype=np.uint8)
    nq = len(lens) * hq * 128
    got = raw[:nq * 4].view(np.float32).reshape(len(lens), hq, 128)
    ntok = raw[nq * 4:].view(np.int64)
    assert ntok.tolist() == lens
    assert np.isfinite(got).all()

    total, longest = sum(lens), max(lens)
    orc = oracle.OraclePool(hkv, total // 32 + 4, total // 32 + 2 * len(lens) + longest // 32 + 8, len(lens),
                            longest // 32 + 8)
    ids = [orc.open() for _ in lens]
    for i, (b, k, v) in enumerate(zip(bits, ks, vs)):
        assert orc.append(np.full(b.size, ids[i], np.int32), b, k, v) == oracle.OK
    assert orc.evict(np.array(ids, np.int32)[ev_req], ev_pos) == oracle.OK
    assert orc.reorder(ids) == oracle.OK
    ref = orc.decode(q, ids, float(scale)).reshape(len(lens), hq, 128)
    assert_outputs_close(got, ref, "C client")
