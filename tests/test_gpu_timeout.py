"""The bounded-wait failure path on the GPU, without a fault: every copy wait in
the scans has an iteration bound, after which the warp records a timeout
status, waits (bounded) for the copies it issued and exits.  kv_set_wait_limit
shortens only the first copy wait of the page scan and of the full-precision
list scan to zero polls, so the wait gives up while the copy is still in
flight; kv_pool_sync must report KV_ERR_DEVICE_TIMEOUT once, clear it, and
leave the pool and the context usable."""
import numpy as np
import pytest

import kvsynth
import oracle
from test_gpu_parity import SCALE, SEED, Scenario, _mixed

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_kv_gb300 as m
    m.load_library()
    return m


def _dev(bits_u16):
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("lists", [False, True])
def test_expired_wait_reports_timeout_once(kvq, lists):
    bits = [_mixed(400, 0.6, 11), _mixed(150, 0.5, 12)]
    sc = Scenario(kvq, 2, 8, bits, chunk=128, impl=2)
    if lists:
        sc.gpu.fp_configure(64)
        for r, (g, o) in enumerate(zip(sc.g_ids, sc.o_ids)):
            k = kvsynth.fill_bf16_host(40, 2, 128, SEED, kvsynth.TENSOR_K, 300 + r)
            v = kvsynth.fill_bf16_host(40, 2, 128, SEED, kvsynth.TENSOR_V, 300 + r)
            sc.gpu.fp_append(g, _dev(k), _dev(v))
            assert sc.orc.fp_append(o, k, v) == oracle.OK
    sc.check_decode(what="before the timeout")
    B = len(sc.g_ids)
    qd = torch.empty((B, 8, 128), dtype=torch.bfloat16, device="cuda")
    kvsynth.fill_bf16_dev(qd.data_ptr(), B, 8, 128, SEED, kvsynth.TENSOR_Q, 1)
    sc.gpu.set_wait_limit(0)
    sc.gpu.decode(qd, sc.g_ids, SCALE)
    with pytest.raises(kvq.KVError) as e:
        sc.gpu.sync()
    assert e.value.status == kvq.KV_ERR_DEVICE_TIMEOUT
    sc.gpu.sync()                                            # reported once, then cleared
    sc.gpu.set_wait_limit(-1)
    sc.check_decode(step=2, what="after the timeout")        # same pool, same context
    with pytest.raises(kvq.KVError) as e:
        sc.gpu.set_wait_limit(-2)
    assert e.value.status == kvq.KV_ERR_INVALID_ARG
