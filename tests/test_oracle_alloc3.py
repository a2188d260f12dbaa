"""Pins of the oracle's greedy allocation over three widths (reading of
TriAxialKV, key design 2, with INT3 from its limitations and outlook): every
tag starts at 2 bits; one-bit steps 2 -> 3 and 3 -> 4 are taken best saving
per bit-token first, a step that does not fit being dropped."""
import itertools

import numpy as np

from conftest import golden_lines


def _ints(f):
    return [int(v) for v in f.split(",")]


def _floats(f):
    return [float(v) for v in f.split(",")]


def test_golden_cases(orc):
    n = 0
    for ln in golden_lines("alloc3_cases.txt"):
        N, D2, D3, D4, B, bits = [f.strip() for f in ln.split("|")]
        bn, bd = map(int, B.split())
        got = orc.alloc_bits3(_ints(N), _floats(D2), _floats(D3), _floats(D4), (bn, bd))
        assert got.tolist() == _ints(bits), ln
        n += 1
    assert n == 4


def _instance(rng, n, equal_n=False, convex=True):
    N = np.full(n, int(rng.integers(1, 50))) if equal_n else rng.integers(0, 200, n)
    D4 = rng.uniform(0.01, 1, n)
    D2 = D4 * (1 + rng.uniform(0.5, 20, n))
    f = rng.uniform(0.2, 0.5, n) if convex else rng.uniform(0.0, 1.0, n)
    D3 = D4 + (D2 - D4) * f          # convex when the 2 -> 3 saving is the larger
    return N.astype(np.int64), D2, D3, D4


def test_budget_feasible_and_maximal(orc):
    """sum N b <= B sum N, and no tag below 4 bits could take its next step."""
    rng = np.random.default_rng(6)
    for _ in range(300):
        n = int(rng.integers(1, 57))
        N, D2, D3, D4 = _instance(rng, n, convex=bool(rng.integers(0, 2)))
        B = (int(rng.integers(20, 41)), 10)
        b = orc.alloc_bits3(N, D2, D3, D4, B).astype(np.int64)
        assert set(b.tolist()) <= {2, 3, 4}
        total = int(N.sum())
        used = int((N * b).sum())
        assert used * B[1] <= B[0] * total
        for k in range(n):
            if b[k] < 4 and N[k] > 0:
                assert (used + N[k]) * B[1] > B[0] * total


def test_optimal_for_equal_counts_and_convex_savings(orc):
    """With equal N_k every step costs the same, so the budget admits a fixed
    number of steps; with each tag's first step saving at least its second,
    the best steps are always takeable in order, and the greedy reaches the
    brute-force minimum of sum N D(b) over all 3^n assignments."""
    rng = np.random.default_rng(7)
    for _ in range(60):
        n = int(rng.integers(1, 7))
        N, D2, D3, D4 = _instance(rng, n, equal_n=True, convex=True)
        B = (int(rng.integers(20, 41)), 10)
        D = np.stack([D2, D3, D4], 1)
        b = orc.alloc_bits3(N, D2, D3, D4, B)
        got = float(sum(N[k] * D[k, b[k] - 2] for k in range(n)))
        total = int(N.sum())
        best = min(float(sum(N[k] * D[k, c[k]] for k in range(n)))
                   for c in itertools.product(range(3), repeat=n)
                   if sum(N[k] * (c[k] + 2) for k in range(n)) * B[1] <= B[0] * total)
        assert abs(got - best) <= 1e-9 * max(1.0, best)


def test_two_way_reduction(orc):
    """When every tag's INT3 saving is exactly half its INT4 saving (D3 =
    (D2 + D4) / 2), both of a tag's steps save the two-way rule's amount per
    bit-token, so they are taken back to back in the two-way order; with equal
    counts and room for exactly k whole upgrades, the allocation equals the
    two-way greedy's (key design 2)."""
    rng = np.random.default_rng(8)
    for _ in range(100):
        n = int(rng.integers(1, 20))
        N = np.full(n, 10, np.int64)
        D4 = rng.uniform(0.01, 1, n)
        D2 = D4 * (1 + rng.uniform(0.5, 20, n))
        D3 = (D2 + D4) / 2
        k4 = int(rng.integers(0, n + 1))
        B = (2 * n + 2 * k4, n)                    # room for exactly k4 two-bit upgrades
        b3 = orc.alloc_bits3(N, D2, D3, D4, B)
        b2 = orc.alloc_bits(N, D2, D4, B)
        assert np.array_equal(b3, b2)
        assert int((b3 == 4).sum()) == k4
