"""kv_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory while decoding (their memory belongs to another
allocator or a fixed budget, or a cudaMalloc would stall a latency-critical
loop).  It must give the same outputs as kv_decode_attn, call after call, using
only the library's fixed internal scratch, and both must match the fp64
oracle.  This file is collected last."""
import numpy as np
import pytest

import kvsynth
import oracle
from harness import OracleWorkload, assert_outputs_close

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
    from mixed_precision_kv_gb300.workload import GPUWorkload, pool_size
    w = kvsynth.make_workload(3, n_req=3, ctx=5000)          # g = 8, INT2 and INT4 pages, x8 rows
    gw = GPUWorkload(w, chunk=2048)
    gw.pool.set_decode_impl(impl)
    ow = OracleWorkload(w, pool_size(w, gw.bits, 2048, gw.steps), 2048)
    for o in (gw, ow):
        o.prefill()
        o.reorder()
    gw.pool.sync()
    for step in (0, 1):                                       # two calls in a row
        q = gw.q(step)
        ref = gw.decode(q).clone()
        out = torch.full_like(ref, float("nan"))
        gw.pool.decode_noalloc(q, gw.rids, w.softmax_scale, out)
        gw.pool.sync()
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        assert_outputs_close(got, ref.cpu().numpy(), f"noalloc vs decode, call {step}")
        orc = ow.decode(ow.q(step)).reshape(got.shape)
        assert_outputs_close(got, orc, f"noalloc vs oracle, call {step}")


@pytest.mark.parametrize("impl", [2, 1])
def test_noalloc_decode_with_int3_and_fp4_pages(kvq, impl):
    """The same two-call comparison on a pool that also holds INT3 and FP4
    pages (the scan variant that reads them)."""
    from mixed_precision_kv_gb300.workload import GPUWorkload, int3_pages, pool_size
    w = kvsynth.make_workload(3, n_req=3, ctx=5000)
    gw = GPUWorkload(w, chunk=2048, int3_share=0.4, fp4_share=0.4)
    gw.pool.set_decode_impl(impl)
    n3, nf = int3_pages(w, gw.bits, gw.steps), int3_pages(w, gw.bits, gw.steps, 0xF4)
    assert n3 > 0 and nf > 0
    ow = OracleWorkload(w, pool_size(w, gw.bits, 2048, gw.steps), 2048, n_int3_pages=n3, n_fp4_pages=nf,
                        int3_share=0.4, fp4_share=0.4)
    for o in (gw, ow):
        o.prefill()
        o.reorder()
    gw.pool.sync()
    for step in (0, 1):
        q = gw.q(step)
        ref = gw.decode(q).clone()
        out = torch.full_like(ref, float("nan"))
        gw.pool.decode_noalloc(q, gw.rids, w.softmax_scale, out)
        gw.pool.sync()
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        assert_outputs_close(got, ref.cpu().numpy(), f"noalloc vs decode with INT3/FP4, call {step}")
        orc = ow.decode(ow.q(step)).reshape(got.shape)
        assert_outputs_close(got, orc, f"noalloc vs oracle with INT3/FP4, call {step}")


def _many_short_requests(kvq, n_req, hkv=8, hq=64, n_tok=70, fp_tokens=2):
    """n_req requests of n_tok mixed INT2/INT4 tokens on both sides, every
    request with `fp_tokens` full-precision list tokens per kv head."""
    from test_gpu_parity import SEED, Scenario, _mixed
    bits = [_mixed(n_tok, 0.6, 1000 + r) for r in range(n_req)]
    sc = Scenario(kvq, hkv, hq, bits, chunk=n_tok)
    sc.gpu.fp_configure(4)
    for r, (g, o) in enumerate(zip(sc.g_ids, sc.o_ids)):
        k = kvsynth.fill_bf16_host(fp_tokens, hkv, 128, SEED, kvsynth.TENSOR_K, 5000 + r)
        v = kvsynth.fill_bf16_host(fp_tokens, hkv, 128, SEED, kvsynth.TENSOR_V, 5000 + r)
        as_dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        sc.gpu.fp_append(g, as_dev(k), as_dev(v))
        assert sc.orc.fp_append(o, k, v) == oracle.OK
    sc.gpu.sync()
    return sc


def test_noalloc_capped_worker_plan(kvq):
    """300 requests at g = 8 with full-precision lists: the per-unit q operands
    (8416 bytes per unit) and the full-precision splits leave room in the
    64 MiB scratch for fewer split partials than the SM count x 16 workers the
    decode plans with, so the entry point plans with fewer workers.  Outputs
    against kv_decode_attn and the oracle, on two calls in a row."""
    from test_gpu_parity import SCALE, SEED
    n_req, hkv, hq = 300, 8, 64
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    units = n_req * hkv
    part = (hq // hkv) * 132 * 4
    budget = ((64 << 20) - units * 32 - units * 8416 - 1024) // (32 + 4 + part)
    assert budget - units - 2 * (sm * 8 + units) < sm * 16, "this case no longer reaches the worker cap"
    sc = _many_short_requests(kvq, n_req, hkv, hq)
    for step in (0, 1):
        qd = torch.empty((n_req, hq, 128), dtype=torch.bfloat16, device="cuda")
        kvsynth.fill_bf16_dev(qd.data_ptr(), n_req, hq, 128, SEED, kvsynth.TENSOR_Q, step)
        ref = sc.gpu.decode(qd, sc.g_ids, SCALE).clone()
        out = torch.full_like(ref, float("nan"))
        sc.gpu.decode_noalloc(qd, sc.g_ids, SCALE, out)
        sc.gpu.sync()
        got = out.cpu().numpy()
        assert np.isfinite(got).all()
        assert_outputs_close(got, ref.cpu().numpy(), f"capped noalloc vs decode, call {step}")
        qh = kvsynth.fill_bf16_host(n_req, hq, 128, SEED, kvsynth.TENSOR_Q, step)
        orc = sc.orc.decode(qh, sc.o_ids, SCALE).reshape(got.shape)
        assert_outputs_close(got, orc, f"capped noalloc vs oracle, call {step}")


def test_noalloc_rejects_plan_that_does_not_fit(kvq):
    """400 requests at g = 8 with full-precision lists (3200 units, under the
    4096-unit limit): the q operands and full-precision splits alone exceed
    the scratch, so the call fails before any device work and `out` keeps
    its contents."""
    from test_gpu_parity import SCALE
    n_req, hq = 400, 64
    sc = _many_short_requests(kvq, n_req, 8, hq, n_tok=40, fp_tokens=1)
    q = torch.zeros((n_req, hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.full((n_req, hq, 128), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(kvq.KVError) as e:
        sc.gpu.decode_noalloc(q, sc.g_ids, SCALE, out)
    assert e.value.status == kvq.KV_ERR_INVALID_ARG
    assert "does not fit" in str(e.value)
    sc.gpu.sync()
    assert bool((out == 7.0).all())


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


def test_noalloc_rejects_tensors_off_the_pool_device(kvq):
    pool = kvq.KVPool(2, 4, 8, 2, 4)
    rid = pool.open()
    q = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        pool.decode_noalloc(q, [rid], 0.1, torch.zeros((1, 8, 128), dtype=torch.float32))   # host out
    with pytest.raises(ValueError):
        pool.decode_noalloc(q.cpu(), [rid], 0.1, torch.zeros((1, 8, 128), dtype=torch.float32, device="cuda"))
