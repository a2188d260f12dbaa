"""Pins of the oracle's greedy INT2/INT4 bit allocator (TriAxialKV, key design 2)."""
import itertools

import numpy as np

from conftest import golden_lines


def _ints(f):
    return [int(v) for v in f.split(",")]


def test_golden_cases(orc):
    n = 0
    for ln in golden_lines("alloc_cases.txt"):
        N, D2, D4, B, bits = [f.strip() for f in ln.split("|")]
        bn, bd = map(int, B.split())
        got = orc.alloc_bits(_ints(N), [float(v) for v in D2.split(",")], [float(v) for v in D4.split(",")],
                             (bn, bd))
        assert got.tolist() == _ints(bits), ln
        n += 1
    assert n == 4


def _instance(rng, n, equal_n=False):
    N = np.full(n, int(rng.integers(1, 50))) if equal_n else rng.integers(0, 200, n)
    D4 = rng.uniform(0.01, 1, n)
    D2 = D4 * (1 + rng.uniform(0.5, 20, n))
    return N.astype(np.int64), D2, D4


def test_budget_feasible_and_maximal(orc):
    """The allocation meets sum N b <= B sum N, and no tag left at 2 bits could
    still be raised to 4 without breaking it (skip-and-continue scan)."""
    rng = np.random.default_rng(5)
    for _ in range(400):
        n = int(rng.integers(1, 57))
        N, D2, D4 = _instance(rng, n)
        B = (int(rng.integers(20, 41)), 10)
        b = orc.alloc_bits(N, D2, D4, B).astype(np.int64)
        total = int(N.sum())
        used = int((N * b).sum())
        assert set(b.tolist()) <= {2, 4}
        assert used * B[1] <= B[0] * total
        for k in range(n):
            if b[k] == 2 and N[k] > 0:
                assert (used + 2 * N[k]) * B[1] > B[0] * total
        assert (b[N == 0] == 2).all()


def test_equal_counts_greedy_is_optimal(orc):
    """With all N_k equal every upgrade costs the same, so ranking by rho is the
    exact optimum of min sum D_k(b_k) under the budget: compare against brute
    force over all 2^|S| assignments."""
    rng = np.random.default_rng(6)
    for _ in range(60):
        n = int(rng.integers(1, 11))
        N, D2, D4 = _instance(rng, n, equal_n=True)
        B = (int(rng.integers(20, 41)), 10)
        b = orc.alloc_bits(N, D2, D4, B)
        obj = float(np.where(b == 4, D4, D2).sum())
        best = np.inf
        for assign in itertools.product((2, 4), repeat=n):
            a = np.array(assign)
            if int((N * a).sum()) * B[1] <= B[0] * int(N.sum()):
                best = min(best, float(np.where(a == 4, D4, D2).sum()))
        assert abs(obj - best) <= 1e-12 * max(1.0, best)


def test_general_counts_never_beats_brute_force_and_picks_top_rho_first(orc):
    rng = np.random.default_rng(7)
    for _ in range(60):
        n = int(rng.integers(2, 11))
        N, D2, D4 = _instance(rng, n)
        N[N == 0] = 1
        B = (int(rng.integers(25, 36)), 10)
        b = orc.alloc_bits(N, D2, D4, B)
        obj = float(np.where(b == 4, D4, D2).sum())
        best = min(float(np.where(np.array(a) == 4, D4, D2).sum())
                   for a in itertools.product((2, 4), repeat=n)
                   if int((N * np.array(a)).sum()) * B[1] <= B[0] * int(N.sum()))
        assert obj >= best - 1e-12
        rho = (D2 - D4) / (2 * N)
        top = int(np.argmax(rho))
        fits_alone = (2 * N.sum() + 2 * N[top]) * B[1] <= B[0] * N.sum()
        assert (b[top] == 4) == bool(fits_alone)
