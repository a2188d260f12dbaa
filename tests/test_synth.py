"""Pins of the seeded input generator (kvsynth) -- not of the method."""
import numpy as np

import kvsynth
from conftest import golden_lines


def test_philox_known_answers():
    rows = [list(map(lambda s: int(s, 16), ln.split())) for ln in golden_lines("philox4x32_10_kat.txt")]
    ctr = np.array([r[0:4] for r in rows], dtype=np.uint32)
    key = np.array([r[4:6] for r in rows], dtype=np.uint32)
    want = np.array([r[6:10] for r in rows], dtype=np.uint32)
    assert (kvsynth.philox_blocks_host(ctr, key) == want).all()
    assert (kvsynth.philox_blocks_np(ctr, key) == want).all()


def test_host_c_matches_numpy_philox_on_random_counters():
    rng = np.random.default_rng(7)
    ctr = rng.integers(0, 2**32, size=(4096, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2**32, size=(4096, 2), dtype=np.uint64).astype(np.uint32)
    assert (kvsynth.philox_blocks_host(ctr, key) == kvsynth.philox_blocks_np(ctr, key)).all()


def test_values_are_irwin_hall_normal_and_multipliers_exact():
    x = kvsynth.bf16_to_f32(kvsynth.fill_bf16_host(512, 4, 128, 1234, kvsynth.TENSOR_K, 3))
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01
    assert float(np.abs(x).max()) <= 6.0
    cm = np.ones((4, 128), np.float32)
    cm[1, 5] = 20.0
    rm = np.ones(512, np.float32)
    rm[7] = 8.0
    y = kvsynth.bf16_to_f32(kvsynth.fill_bf16_host(512, 4, 128, 1234, kvsynth.TENSOR_K, 3,
                                                   chan_mult=cm, row_mult=rm))
    base = x.astype(np.float64) * cm[None].astype(np.float64) * rm[:, None, None]
    # the multipliers act on the fp32 draw before its bf16 rounding (x8 is exact)
    assert np.array_equal(y[:, 0], x[:, 0] * rm[:, None])
    assert np.allclose(y, base, rtol=2 ** -7, atol=0)


def test_offsets_compose():
    a = kvsynth.fill_bf16_host(40, 2, 128, 99, kvsynth.TENSOR_V, 5)
    b = kvsynth.fill_bf16_host(15, 2, 128, 99, kvsynth.TENSOR_V, 5, tok0=25)
    assert np.array_equal(a[25:], b)


def test_workload_recipes_shapes():
    w = kvsynth.make_workload(4)
    assert len(w.requests) == 64 and w.g == 4
    for r in w.requests:
        assert 1024 <= r.n_prefill <= 131072
        assert r.tags.size == r.n_prefill and r.tags.max() < 56
        assert r.evict.size == round(0.05 * r.n_prefill)
        assert 2.2 <= r.budget[0] / r.budget[1] <= 3.6
    w3 = kvsynth.make_workload(3, n_req=2, ctx=1000)
    assert (w3.requests[0].row_mult == 8).sum() == 10
    assert (w3.k_chan_mult == 20).sum(axis=1).tolist() == [4] * 8
