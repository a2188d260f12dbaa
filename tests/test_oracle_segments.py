"""Pins of the oracle's full-precision segments and per-head exclusion
(HyQuant, core method: K = K_VL u K_Win u K_Q, mutually exclusive per head;
Algorithm 3: the quantized prefix, then the vertical-line, staging and window
tokens under one online-softmax state)."""
import numpy as np
import pytest

import kvsynth

SCALE = float(np.float32(1 / np.sqrt(128)))


def _bf16(x):
    """float32 values that bf16 holds exactly -> bf16 bits."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32)
    assert not np.any(b & 0xFFFF), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def _q(B, Hq, seed=9):
    return kvsynth.fill_bf16_host(B, Hq, 128, seed, kvsynth.TENSOR_Q, 0)


def _rows(n, hkv, tensor, seed=3, stream=0):
    return kvsynth.fill_bf16_host(n, hkv, 128, seed, tensor, stream)


def test_single_fp_token_returns_its_value_per_head(orc):
    """One token and nothing else: softmax weight 1, the output is that head's
    own V row (distinct rows per head catch a head-index mix-up)."""
    hkv, g = 4, 2
    P = orc.OraclePool(hkv, 8, 8, 2, 8)
    r = P.open()
    k, v = _rows(1, hkv, kvsynth.TENSOR_K), _rows(1, hkv, kvsynth.TENSOR_V)
    assert P.fp_append(r, k, v) == orc.OK
    out = P.decode(_q(1, hkv * g), [r], SCALE)
    for hq in range(hkv * g):
        np.testing.assert_array_equal(out[hq], kvsynth.bf16_to_f32(v[0, hq // g]).astype(np.float64))


def test_two_fp_tokens_closed_form(orc):
    """Two tokens: the output is s v1 + (1 - s) v2 with s the logistic of
    scale * q . (k1 - k2)."""
    hkv, g = 1, 4
    P = orc.OraclePool(hkv, 8, 8, 1, 8)
    r = P.open()
    rng = np.random.default_rng(2)
    kf = rng.integers(-4, 5, (2, hkv, 128)).astype(np.float32) / 4
    vf = rng.integers(-8, 9, (2, hkv, 128)).astype(np.float32) / 8
    assert P.fp_append(r, _bf16(kf), _bf16(vf)) == orc.OK
    q = _q(1, g)
    out = P.decode(q, [r], SCALE)
    for hq in range(g):
        qd = kvsynth.bf16_to_f32(q[0, hq]).astype(np.float64)
        d = SCALE * float(qd @ (kf[0, 0].astype(np.float64) - kf[1, 0]))
        s = 1.0 / (1.0 + np.exp(-d))
        np.testing.assert_allclose(out[hq], s * vf[0, 0] + (1 - s) * vf[1, 0], rtol=1e-12, atol=1e-14)


def test_fp_only_is_plain_softmax_attention(orc):
    """A request whose tokens are all full precision: textbook softmax
    attention over the bf16 rows; split invariance holds."""
    hkv, g, n = 2, 4, 300
    P = orc.OraclePool(hkv, 8, 8, 1, 8)
    r = P.open()
    k, v = _rows(n, hkv, kvsynth.TENSOR_K), _rows(n, hkv, kvsynth.TENSOR_V)
    assert P.fp_append(r, k[:100], v[:100]) == orc.OK
    assert P.fp_append(r, k[100:], v[100:]) == orc.OK
    q = _q(1, hkv * g)
    out = P.decode(q, [r], SCALE)
    for hq in range(hkv * g):
        K = kvsynth.bf16_to_f32(k[:, hq // g]).astype(np.float64)
        V = kvsynth.bf16_to_f32(v[:, hq // g]).astype(np.float64)
        lg = SCALE * (K @ kvsynth.bf16_to_f32(q[0, hq]).astype(np.float64))
        w = np.exp(lg - lg.max())
        np.testing.assert_allclose(out[hq], (w @ V) / w.sum(), rtol=1e-12, atol=1e-14)
    for s in (2, 7, 301):
        np.testing.assert_allclose(P.decode(q, [r], SCALE, n_splits=s), out, rtol=1e-12, atol=1e-14)


def _exact_values(n, hkv, seed):
    """Rows whose quantization is exact at both widths: values c * {0, 5, 10,
    15} with c = 1/8, each 32-channel group of a token and each channel of
    every 32-token page holding both 0 and 15 c.  INT4 then has s = c, z = 0,
    INT2 (K per channel, V per token) s = 5c, z = 0: every dequantized value
    is the input value."""
    rng = np.random.default_rng(seed)
    lv = rng.integers(0, 4, (n, hkv, 128)) * 5
    t = np.arange(n)[:, None]
    c = np.arange(128)[None, :]
    # token t: channel (t mod 32) of every group is 0, channel ((t + 16) mod 32) is 15
    # -> per token group: 0 and 15 present; per channel: over 32 tokens both occur
    zero = (c % 32) == (t % 32)
    full = (c % 32) == ((t + 16) % 32)
    for h in range(hkv):
        lv[:, h][zero] = 0
        lv[:, h][full] = 15
    return _bf16(lv.astype(np.float32) / 8)


@pytest.mark.parametrize("n", [130, 200])
def test_fp_copy_replaces_quantized_copy_exactly(orc, n):
    """Each head moves its own position from the quantized set to the
    full-precision list (per-head exclusion + one full-precision token holding
    that head's row).  With exactly quantizable values the token set of every
    head is unchanged, so the output is too (up to summation order).  Two of
    the exclusions hit INT2-tagged tokens still waiting in their staging page,
    so the exclusion must survive the requantization into the INT2 page."""
    hkv, g = 3, 2
    k, v = _exact_values(n, hkv, 1), _exact_values(n, hkv, 2)
    bits = np.where(np.random.default_rng(4).random(n) < 0.6, 2, 4).astype(np.uint8)
    q = _q(1, hkv * g)
    A = orc.OraclePool(hkv, 64, 64, 1, 64)
    ra = A.open()
    assert A.append(np.full(n, ra), bits, k, v) == orc.OK
    base = A.decode(q, [ra], SCALE)
    # the values quantize exactly: the pool's output is attention over the inputs
    for hq in range(hkv * g):
        K = kvsynth.bf16_to_f32(k[:, hq // g]).astype(np.float64)
        V = kvsynth.bf16_to_f32(v[:, hq // g]).astype(np.float64)
        lg = SCALE * (K @ kvsynth.bf16_to_f32(q[0, hq]).astype(np.float64))
        w = np.exp(lg - lg.max())
        np.testing.assert_allclose(base[hq], (w @ V) / w.sum(), rtol=1e-12, atol=1e-14)

    half = n // 2
    idx2 = np.flatnonzero(bits[:half] == 2)
    staged = idx2[idx2.size - idx2.size % 32:]          # INT2-tagged, still in the staging page
    assert staged.size >= 2 and staged.size + np.count_nonzero(bits[half:] == 2) >= 32
    pos = np.array([staged[-1], staged[0], np.flatnonzero(bits[:half] == 4)[0]])   # one per kv head
    B = orc.OraclePool(hkv, 64, 64, 1, 64)
    rb = B.open()
    assert B.append(np.full(half, rb), bits[:half], k[:half], v[:half]) == orc.OK
    assert B.evict_head(np.full(hkv, rb), pos, np.arange(hkv)) == orc.OK
    assert B.append(np.full(n - half, rb), bits[half:], k[half:], v[half:]) == orc.OK
    kf = np.stack([k[pos[h], h] for h in range(hkv)])[None]
    vf = np.stack([v[pos[h], h] for h in range(hkv)])[None]
    assert B.fp_append(rb, kf, vf) == orc.OK
    np.testing.assert_allclose(B.decode(q, [rb], SCALE), base, rtol=1e-12, atol=1e-14)
    # without the exclusion the moved token counts twice: the output changes
    C = orc.OraclePool(hkv, 64, 64, 1, 64)
    rc = C.open()
    assert C.append(np.full(n, rc), bits, k, v) == orc.OK
    assert C.fp_append(rc, kf, vf) == orc.OK
    assert np.abs(C.decode(q, [rc], SCALE) - base).max() > 1e-6


def test_head_exclusion_for_every_head_equals_eviction(orc):
    rng = np.random.default_rng(7)
    hkv, n = 2, 150
    k, v = _rows(n, hkv, kvsynth.TENSOR_K), _rows(n, hkv, kvsynth.TENSOR_V)
    bits = np.where(rng.random(n) < 0.5, 2, 4).astype(np.uint8)
    ev = rng.choice(n, 20, replace=False)
    q = _q(1, 8)
    A = orc.OraclePool(hkv, 64, 64, 1, 64)
    ra = A.open()
    assert A.append(np.full(n, ra), bits, k, v) == orc.OK
    assert A.evict(np.full(ev.size, ra), ev) == orc.OK
    B = orc.OraclePool(hkv, 64, 64, 1, 64)
    rb = B.open()
    assert B.append(np.full(n, rb), bits, k, v) == orc.OK
    for h in range(hkv):
        assert B.evict_head(np.full(ev.size, rb), ev, np.full(ev.size, h)) == orc.OK
    np.testing.assert_array_equal(B.decode(q, [rb], SCALE), A.decode(q, [ra], SCALE))
    # one head only: the other head's outputs are those of the uncut pool
    C = orc.OraclePool(hkv, 64, 64, 1, 64)
    rc = C.open()
    assert C.append(np.full(n, rc), bits, k, v) == orc.OK
    full = C.decode(q, [rc], SCALE)
    assert C.evict_head(np.full(ev.size, rc), ev, np.zeros(ev.size)) == orc.OK
    cut = C.decode(q, [rc], SCALE)
    np.testing.assert_array_equal(cut[4:], full[4:])
    np.testing.assert_array_equal(cut[:4], A.decode(q, [ra], SCALE)[:4])


def test_drop_keeps_order_of_the_rest(orc):
    hkv, n = 2, 40
    k, v = _rows(n, hkv, kvsynth.TENSOR_K), _rows(n, hkv, kvsynth.TENSOR_V)
    q = _q(1, 4)
    A = orc.OraclePool(hkv, 8, 8, 1, 8)
    ra = A.open()
    assert A.fp_append(ra, k, v) == orc.OK
    assert A.fp_drop(ra, 10, 5) == orc.OK
    assert A.fp_drop(ra, 0, 0) == orc.OK
    B = orc.OraclePool(hkv, 8, 8, 1, 8)
    rb = B.open()
    keep = np.r_[0:10, 15:n]
    assert B.fp_append(rb, k[keep], v[keep]) == orc.OK
    np.testing.assert_array_equal(A.decode(q, [ra], SCALE), B.decode(q, [rb], SCALE))
    assert A.fp_drop(ra, 30, 6) == orc.INVALID       # past the end
    assert A.fp_drop(ra, -1, 1) == orc.INVALID
    assert A.evict_head([ra], [0], [0]) == orc.INVALID   # no quantized token at 0
    assert A.fp_drop(ra, 0, n - 5) == orc.OK
    np.testing.assert_array_equal(A.decode(q, [ra], SCALE), np.zeros((4, 128)))


def test_mixed_request_split_invariance(orc):
    """Quantized tokens, per-head exclusions and a full-precision list: the
    split + log-sum-exp merge gives the one-pass result."""
    rng = np.random.default_rng(12)
    hkv, n, nf = 2, 500, 70
    k, v = _rows(n, hkv, kvsynth.TENSOR_K), _rows(n, hkv, kvsynth.TENSOR_V)
    bits = np.where(rng.random(n) < 0.55, 2, 4).astype(np.uint8)
    P = orc.OraclePool(hkv, 64, 64, 1, 64)
    r = P.open()
    assert P.append(np.full(n, r), bits, k, v) == orc.OK
    ex = rng.choice(n, 30, replace=False)
    assert P.evict_head(np.full(ex.size, r), ex, ex % hkv) == orc.OK
    kf, vf = _rows(nf, hkv, kvsynth.TENSOR_K, seed=8), _rows(nf, hkv, kvsynth.TENSOR_V, seed=8)
    assert P.fp_append(r, kf, vf) == orc.OK
    q = _q(1, 8)
    base = P.decode(q, [r], SCALE)
    for s in (2, 5, 64, 1000):
        np.testing.assert_allclose(P.decode(q, [r], SCALE, n_splits=s), base, rtol=1e-12, atol=1e-14)


def test_head_budget_all_excluded_head_reads_zero(orc):
    """Per-head budgets: a head that keeps nothing outputs 0 (every slot is a
    dead slot for it), a head that keeps a suffix equals attention over that
    suffix alone, and the other heads are untouched."""
    rng = np.random.default_rng(31)
    hkv, n = 3, 160
    k, v = _rows(n, hkv, kvsynth.TENSOR_K), _rows(n, hkv, kvsynth.TENSOR_V)
    bits = np.where(rng.random(n) < 0.5, 2, 4).astype(np.uint8)
    q = _q(1, 2 * hkv)
    A = orc.OraclePool(hkv, 64, 64, 1, 64)
    ra = A.open()
    assert A.append(np.full(n, ra), bits, k, v) == orc.OK
    full = A.decode(q, [ra], SCALE)
    cut = 100
    assert A.evict_head(np.full(n, ra), np.arange(n), np.zeros(n)) == orc.OK          # head 0 keeps nothing
    assert A.evict_head(np.full(cut, ra), np.arange(cut), np.ones(cut)) == orc.OK     # head 1 keeps the last 60
    out = A.decode(q, [ra], SCALE)
    np.testing.assert_array_equal(out[0:2], np.zeros((2, 128)))
    np.testing.assert_array_equal(out[4:6], full[4:6])
    # head 1 = the same pool with the first `cut` positions evicted for every head
    B = orc.OraclePool(hkv, 64, 64, 1, 64)
    rb = B.open()
    assert B.append(np.full(n, rb), bits, k, v) == orc.OK
    assert B.evict(np.full(cut, rb), np.arange(cut)) == orc.OK
    np.testing.assert_array_equal(out[2:4], B.decode(q, [rb], SCALE)[2:4])
