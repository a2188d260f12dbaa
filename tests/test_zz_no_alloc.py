"""kv_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory while decoding (their memory belongs to another
allocator or a fixed budget, or a cudaMalloc would stall a latency-critical
loop).  It must give the same outputs as kv_decode_attn, call after call, using
only the library's fixed internal scratch.  This file is collected last."""
import numpy as np
import pytest

import kvsynth
from harness import assert_outputs_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import mixed_precision_kv_gb300 as m
    m.load_library()
    return m


@pytest.mark.parametrize("impl", [2, 1])
def test_noalloc_decode_matches_decode_on_two_calls(kvq, impl):
    from mixed_precision_kv_gb300.workload import GPUWorkload
    w = kvsynth.make_workload(3, n_req=3, ctx=5000)          # g = 8, INT2 and INT4 pages, x8 rows
    gw = GPUWorkload(w, chunk=2048)
    gw.pool.set_decode_impl(impl)
    gw.prefill()
    gw.reorder()
    gw.pool.sync()
    for step in (0, 1):                                       # two calls in a row
        q = gw.q(step)
        ref = gw.decode(q).clone()
        out = torch.full_like(ref, float("nan"))
        gw.pool.decode_noalloc(q, gw.rids, w.softmax_scale, out)
        gw.pool.sync()
        assert torch.isfinite(out).all()
        assert_outputs_close(out.cpu().numpy(), ref.cpu().numpy(), f"noalloc call {step}")


def test_noalloc_rejects_plans_beyond_its_scratch(kvq):
    pool = kvq.KVPool(8, 4, 8, 600, 4)
    rids = [pool.open() for _ in range(513)]                  # 513 x 8 = 4104 units > 4096
    q = torch.zeros((513, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((513, 8, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(kvq.KVError) as e:
        pool.decode_noalloc(q, rids, 0.1, out)
    assert e.value.status == kvq.KV_ERR_INVALID_ARG
    assert "4096" in str(e.value)
    assert np.array_equal(out.cpu().numpy(), np.zeros((513, 8, 128), np.float32))
