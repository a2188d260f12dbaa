"""CUDA path vs oracle with HyQuant full-precision segments and per-head
exclusion: each head moves its own (vertical-line) positions out of the
quantized set into its full-precision list, the window tokens follow; outputs
within max-abs 1e-3 and relative-L2 1e-4 of the fp64 oracle."""
import numpy as np
import pytest

import kvsynth
import oracle
from test_gpu_parity import IMPLS, SCALE, SEED, Scenario, _mixed

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


def _anchor_rows(sc, r, pos_per_head):
    """K/V rows of each head's own positions (the values the quantized copy was made from)."""
    n = len(pos_per_head[0])
    k = np.zeros((n, sc.hkv, 128), np.uint16)
    v = np.zeros((n, sc.hkv, 128), np.uint16)
    for h, pos in enumerate(pos_per_head):
        for j, p in enumerate(pos):
            k[j, h] = kvsynth.fill_bf16_host(1, sc.hkv, 128, SEED, kvsynth.TENSOR_K, r, int(p))[0, h]
            v[j, h] = kvsynth.fill_bf16_host(1, sc.hkv, 128, SEED, kvsynth.TENSOR_V, r, int(p))[0, h]
    return k, v


def _freeze(sc, rng, rho=0.05, window=0, stream0=100):
    """Per request: every head excludes its own top-rho positions (a seeded
    draw standing in for the column score) and appends their rows to its list,
    then `window` recent tokens (fresh rows) follow in full precision."""
    for r, (g, o) in enumerate(zip(sc.g_ids, sc.o_ids)):
        _, n_tok = sc.orc.info(o)
        n_vl = int(rho * n_tok)
        if n_vl:
            pos = [np.sort(rng.choice(n_tok, n_vl, replace=False)) for _ in range(sc.hkv)]
            req = np.full(n_vl * sc.hkv, g)
            allp = np.concatenate(pos)
            heads = np.repeat(np.arange(sc.hkv), n_vl)
            sc.gpu.evict_head(req, allp, heads)
            assert sc.orc.evict_head(np.full(allp.size, o), allp, heads) == oracle.OK
            k, v = _anchor_rows(sc, r, pos)
            sc.gpu.fp_append(g, _dev(k), _dev(v))
            assert sc.orc.fp_append(o, k, v) == oracle.OK
        if window:
            _append_window(sc, r, window, stream0 + r)


def _append_window(sc, r, n, stream, tok0=0):
    k = kvsynth.fill_bf16_host(n, sc.hkv, 128, SEED, kvsynth.TENSOR_K, stream, tok0)
    v = kvsynth.fill_bf16_host(n, sc.hkv, 128, SEED, kvsynth.TENSOR_V, stream, tok0)
    sc.gpu.fp_append(sc.g_ids[r], _dev(k), _dev(v))
    assert sc.orc.fp_append(sc.o_ids[r], k, v) == oracle.OK


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("hkv,hq", [(2, 8), (1, 8), (4, 8), (2, 2), (64, 512)])
def test_vertical_lines_and_window(kvq, impl, hkv, hq):
    bits = [_mixed(700, 0.6, 1), _mixed(333, 0.4, 2), _mixed(90, 0.7, 3)]
    sc = Scenario(kvq, hkv, hq, bits, chunk=128, impl=impl,
                  evict={0: np.arange(5, 600, 37), 2: np.array([0, 1, 2, 60])})
    sc.gpu.fp_configure(512)
    _freeze(sc, np.random.default_rng(7), rho=0.05, window=130)
    sc.gpu.sync()
    sc.check_decode(what=f"hkv={hkv} hq={hq} impl={impl}")
    # the no-allocation decode plans the same splits
    B = len(sc.g_ids)
    qd = torch.empty((B, hq, 128), dtype=torch.bfloat16, device="cuda")
    kvsynth.fill_bf16_dev(qd.data_ptr(), B, hq, 128, SEED, kvsynth.TENSOR_Q, 0)
    out = torch.empty((B, hq, 128), dtype=torch.float32, device="cuda")
    sc.gpu.decode_noalloc(qd, sc.g_ids, SCALE, out)
    sc.gpu.sync()
    ref = sc.orc.decode(kvsynth.fill_bf16_host(B, hq, 128, SEED, kvsynth.TENSOR_Q, 0), sc.o_ids, SCALE)
    from harness import assert_outputs_close
    assert_outputs_close(out.cpu().numpy(), ref.reshape(B, hq, 128), "noalloc")


@pytest.mark.parametrize("impl", IMPLS)
def test_window_slides_with_plan_reuse(kvq, impl):
    """One decode step at a time: a token enters the window, and every 32
    steps the oldest 32 window tokens leave the list and are appended to the
    quantized pool (the staging buffer flushed).  The plan is reused while the
    lists grow by less than a chunk and rebuilt when they shrink."""
    bits = [_mixed(400, 0.6, 4), _mixed(150, 0.5, 5)]
    sc = Scenario(kvq, 2, 8, bits, chunk=96, impl=impl)
    sc.gpu.fp_configure(256)
    _freeze(sc, np.random.default_rng(3), rho=0.05, window=0)
    wpos = [0, 0]
    window = [[], []]   # (stream, tok) of each window token, list order
    for step in range(70):
        for r in range(2):
            _append_window(sc, r, 1, 200 + r, wpos[r])
            window[r].append(wpos[r])
            wpos[r] += 1
        if step % 32 == 31:
            for r, (g, o) in enumerate(zip(sc.g_ids, sc.o_ids)):
                n_fp = sc.gpu.fp_count(g)
                first = n_fp - len(window[r])      # the window follows the vertical lines
                sc.gpu.fp_drop(g, first, 32)
                assert sc.orc.fp_drop(o, first, 32) == oracle.OK
                t0 = window[r][0]
                k = kvsynth.fill_bf16_host(32, 2, 128, SEED, kvsynth.TENSOR_K, 200 + r, t0)
                v = kvsynth.fill_bf16_host(32, 2, 128, SEED, kvsynth.TENSOR_V, 200 + r, t0)
                b = np.full(32, 2, np.uint8)
                sc.gpu.append(_dev(k), _dev(v), np.full(32, g), b)
                assert sc.orc.append(np.full(32, o), b, k, v) == oracle.OK
                window[r] = window[r][32:]
        if step % 7 == 0 or step % 32 == 31:
            sc.check_decode(step=step, what=f"step {step}")


def test_full_precision_only_and_empty(kvq):
    """A request with no quantized token, one with neither, one with both."""
    bits = [np.zeros(0, np.uint8), np.zeros(0, np.uint8), _mixed(64, 0.5, 9)]
    sc = Scenario(kvq, 2, 8, bits, chunk=64)
    sc.gpu.fp_configure(200)
    _append_window(sc, 0, 1, 300)
    sc.check_decode(what="one token")
    _append_window(sc, 0, 199, 301)
    _append_window(sc, 2, 65, 302)
    sc.gpu.sync()
    sc.check_decode(what="fp only / empty / both")


def test_exclusion_follows_repack_and_clears_on_close(kvq):
    """Exclusions on INT2-tagged tokens still in their staging page survive the
    requantization (both the per-token repack and a later bulk call); a closed
    request's exclusions do not leak into the request that reuses its pages."""
    bits = [np.full(20, 2, np.uint8), _mixed(50, 0.5, 11)]
    sc = Scenario(kvq, 2, 8, bits, chunk=64, reorder=False)
    for g, o, pos in zip(sc.g_ids, sc.o_ids, ([3, 19], [0, 49])):
        sc.gpu.evict_head(np.full(2, g), pos, [1, 0])
        assert sc.orc.evict_head(np.full(2, o), pos, [1, 0]) == oracle.OK
    for r, n in ((0, 60), (1, 40)):
        k = kvsynth.fill_bf16_host(n, 2, 128, SEED, kvsynth.TENSOR_K, 50 + r)
        v = kvsynth.fill_bf16_host(n, 2, 128, SEED, kvsynth.TENSOR_V, 50 + r)
        b = _mixed(n, 0.8, 20 + r)
        sc.gpu.append(_dev(k), _dev(v), np.full(n, sc.g_ids[r]), b)
        assert sc.orc.append(np.full(n, sc.o_ids[r]), b, k, v) == oracle.OK
    sc.gpu.sync()
    sc.check_content()
    sc.check_decode(what="after repack")
    # close request 0 and reopen: same page ids, no exclusions
    sc.gpu.close_request(sc.g_ids[0])
    assert sc.orc.close_request(sc.o_ids[0]) is None
    sc.g_ids[0] = sc.gpu.open()
    sc.o_ids[0] = sc.orc.open()
    k = kvsynth.fill_bf16_host(80, 2, 128, SEED, kvsynth.TENSOR_K, 60)
    v = kvsynth.fill_bf16_host(80, 2, 128, SEED, kvsynth.TENSOR_V, 60)
    b = np.full(80, 2, np.uint8)
    sc.gpu.append(_dev(k), _dev(v), np.full(80, sc.g_ids[0]), b)
    assert sc.orc.append(np.full(80, sc.o_ids[0]), b, k, v) == oracle.OK
    sc.gpu.sync()
    sc.check_content()
    sc.check_decode(what="reopened")


def test_list_errors(kvq):
    sc = Scenario(kvq, 2, 4, [_mixed(40, 0.5, 1)], chunk=64)
    g = sc.g_ids[0]
    k = _dev(kvsynth.fill_bf16_host(5, 2, 128, SEED, kvsynth.TENSOR_K, 7))
    with pytest.raises(kvq.KVError):
        sc.gpu.fp_append(g, k, k)          # not configured
    sc.gpu.fp_configure(8)
    sc.gpu.fp_append(g, k, k)
    with pytest.raises(kvq.KVError):
        sc.gpu.fp_append(g, k, k)          # past the capacity
    assert sc.gpu.fp_count(g) == 5
    with pytest.raises(kvq.KVError):
        sc.gpu.fp_drop(g, 3, 3)            # past the end
    with pytest.raises(kvq.KVError):
        sc.gpu.fp_configure(16)            # a list is not empty
    with pytest.raises(kvq.KVError):
        sc.gpu.evict_head([g], [40], [0])  # no token at 40
    with pytest.raises(kvq.KVError):
        sc.gpu.evict_head([g], [0], [2])   # no kv head 2
    sc.gpu.fp_drop(g, 0, 5)
    assert sc.gpu.fp_count(g) == 0
    sc.gpu.fp_configure(16)


def test_batched_append_interleaves_requests(kvq):
    """One kv_fp_append call whose tokens belong to several requests, in mixed
    order: each request's tokens land at the end of its lists, in order."""
    bits = [_mixed(100, 0.5, 1), _mixed(60, 0.5, 2), _mixed(33, 0.5, 3)]
    sc = Scenario(kvq, 2, 8, bits, chunk=64)
    sc.gpu.fp_configure(64)
    _append_window(sc, 1, 5, 400)                  # request 1 already has a list
    order = np.array([0, 1, 0, 2, 1, 0, 0, 2, 1, 1, 0])
    k = kvsynth.fill_bf16_host(order.size, 2, 128, SEED, kvsynth.TENSOR_K, 401)
    v = kvsynth.fill_bf16_host(order.size, 2, 128, SEED, kvsynth.TENSOR_V, 401)
    sc.gpu.fp_append(np.array(sc.g_ids)[order], _dev(k), _dev(v))
    for r in range(3):
        sel = np.flatnonzero(order == r)
        assert sc.orc.fp_append(sc.o_ids[r], k[sel], v[sel]) == oracle.OK
    assert [sc.gpu.fp_count(g) for g in sc.g_ids] == [5, 9, 2]
    sc.gpu.sync()
    sc.check_decode(what="batched append")


@pytest.mark.parametrize("impl", IMPLS)
def test_ragged_head_retention(kvq, impl):
    """Heads keep different amounts of context (a per-head budget): head h
    drops every position before its cut, so whole pages are dead for it and
    the tensor-core scan skips them; one head of one request drops all."""
    bits = [_mixed(900, 0.6, 1), _mixed(400, 0.5, 2)]
    hkv, hq = 4, 16
    sc = Scenario(kvq, hkv, hq, bits, chunk=128, impl=impl)
    for r, (g, o) in enumerate(zip(sc.g_ids, sc.o_ids)):
        n = bits[r].size
        cuts = [0, n // 4, n // 2, n if r == 1 else (7 * n) // 8]
        pos = np.concatenate([np.arange(c) for c in cuts])
        heads = np.concatenate([np.full(c, h) for h, c in enumerate(cuts)])
        sc.gpu.evict_head(np.full(pos.size, g), pos, heads)
        assert sc.orc.evict_head(np.full(pos.size, o), pos, heads) == oracle.OK
    sc.gpu.sync()
    sc.check_decode(what=f"ragged retention impl={impl}")
    stats = sc.gpu.last_decode_stats()
    assert stats["kv_bytes"] > 0
    # appends after the cut are read by every head
    k = kvsynth.fill_bf16_host(40, hkv, 128, SEED, kvsynth.TENSOR_K, 70)
    v = kvsynth.fill_bf16_host(40, hkv, 128, SEED, kvsynth.TENSOR_V, 70)
    b = _mixed(40, 0.5, 71)
    sc.gpu.append(_dev(k), _dev(v), np.full(40, sc.g_ids[1]), b)
    assert sc.orc.append(np.full(40, sc.o_ids[1]), b, k, v) == oracle.OK
    sc.gpu.sync()
    sc.check_decode(step=1, what=f"ragged retention after append impl={impl}")
