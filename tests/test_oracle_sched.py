"""Pins of the scheduler oracle: brute force over every allocation, Algorithm 1
traced by hand, closed-form cost-table values and limiting cases."""
import numpy as np
import pytest

import oracle
import specsynth

COSTS = specsynth.COST_TABLES


# ------------------------------------------------------------------ cost table
@pytest.mark.parametrize("N,expect", [
    (-5.0, 8.0), (0.0, 8.0), (256.0, 8.0 + 256.0 * 10.24 / 512.0), (512.0, 18.24),
    (512.5, 18.24 + 0.5 * 1.76), (513.0, 20.0), (4000.0, 20.0)])
def test_cost_table_bprime_closed_form(N, expect):
    assert abs(oracle.cost_at(N, COSTS["Bprime"]) - expect) < 1e-12


def test_cost_table_readings_A_and_C():
    assert abs(oracle.cost_at(300, COSTS["A"]) - (8 + 0.02 * 300)) < 1e-12
    assert abs(oracle.cost_at(700, COSTS["A"]) - 20.0) < 1e-12
    assert abs(oracle.cost_at(700, COSTS["C"]) - 18.24) < 1e-12


# --------------------------------------------------- Algorithm 1 hand traces
def test_algorithm1_hand_trace_takes_all():
    """R=2, gamma=2, c = [[0.9, 0.5], [0.6, 0.9]] -> survivals r0: [0.9, 0.45],
    r1: [0.6, 0.54]; order 0.9, 0.6, 0.54, 0.45.  With C(N) = 10 + N:
    2/12 < 2.9/13 < 3.5/14 < 4.04/15 < 4.49/16, so every candidate is kept."""
    conf = np.array([[0.9, 0.5], [0.6, 0.9]], np.float32)
    cost = ([0.0, 100.0], [10.0, 110.0])
    r = oracle.sched_alg1(conf, cost)
    assert r["rc"] == 0 and list(r["verify_len"]) == [2, 2]
    e = oracle.sched_exact(conf, cost)
    assert list(e["verify_len"]) == [2, 2]
    assert abs(e["obj"] - 4.49 / 16.0) < 1e-6


def test_algorithm1_hand_trace_stops_first():
    """Same confidences, C(N) = N: 2/2 = 1 > 2.9/3, so the first candidate is
    reverted and every request keeps only its anchor."""
    conf = np.array([[0.9, 0.5], [0.6, 0.9]], np.float32)
    cost = ([1.0, 100.0], [1.0, 100.0])
    assert list(oracle.sched_alg1(conf, cost)["verify_len"]) == [0, 0]
    assert list(oracle.sched_exact(conf, cost)["verify_len"]) == [0, 0]


def test_algorithm1_hand_trace_middle():
    """C(N) = 2 + N: 2/4=.5, 2.9/5=.58, 3.5/6=.5833, 4.04/7=.5771 -> stop after
    the second candidate: r0 keeps depth 1, r1 keeps depth 1."""
    conf = np.array([[0.9, 0.5], [0.6, 0.9]], np.float32)
    cost = ([0.0, 100.0], [2.0, 102.0])
    assert list(oracle.sched_alg1(conf, cost)["verify_len"]) == [1, 1]
    assert list(oracle.sched_exact(conf, cost)["verify_len"]) == [1, 1]


# ------------------------------------------------------------ brute force
@pytest.mark.parametrize("cost_name", ["affine", "Bprime", "A", "C"])
@pytest.mark.parametrize("min_len", [0, 1])
def test_exact_matches_brute_force(cost_name, min_len):
    """sched_exact equals enumeration of every allocation in [min_len, gamma]^B
    for B <= 4, gamma <= 4: 10^4 random confidence draws per cost reading and
    min_len (near-ties within 1e-12 relative are skipped)."""
    rng = np.random.default_rng(10 + min_len)
    kt, kc = COSTS[cost_name]
    checked = 0
    for trial in range(10000):
        B = int(rng.integers(1, 5))
        gamma = int(rng.integers(max(1, min_len), 5))
        conf = rng.uniform(0.0, 1.0, (B, gamma)).astype(np.float32)
        # scale the table so the optimum falls anywhere in [B(min_len+1), B(gamma+1)]
        s = float(rng.uniform(0.002, 0.2))
        cost = (np.array(kt) * s, np.array(kc))
        if cost_name == "affine":
            cost = ([0.0, 10.0], [1.0, 1.0 + 10.0 * float(rng.uniform(0.01, 2.0))])
        e = oracle.sched_exact(conf, cost, min_len)
        b = oracle.sched_brute(conf, cost, min_len)
        assert e["rc"] == 0 and b["rc"] == 0
        if min(e["gap"], b["gap"]) < 1e-12:
            continue
        checked += 1
        assert list(e["verify_len"]) == list(b["verify_len"]), (conf, cost)
        assert abs(e["obj"] - b["obj"]) <= 1e-12 * abs(b["obj"])
    assert checked > 9000


def test_alg1_equals_exact_under_affine_costs():
    rng = np.random.default_rng(3)
    for trial in range(2000):
        B = int(rng.integers(1, 65))
        gamma = int(rng.integers(1, 17))
        conf = specsynth.make_confidences(B, gamma, seed=1000 + trial)
        a, b = float(rng.uniform(0.5, 20)), float(rng.uniform(0.001, 2.0))
        cost = ([0.0, 1e6], [a, a + b * 1e6])
        e = oracle.sched_exact(conf, cost, 1 if trial % 2 else 0)
        g = oracle.sched_alg1(conf, cost, 1 if trial % 2 else 0)
        assert list(e["verify_len"]) == list(g["verify_len"])


def test_alg1_can_stop_early_under_flat_cost():
    """Reading C (cost flat beyond 512) makes tau/C non-concave: the exact scan
    verifies everything while Algorithm 1 stops at its first non-improvement."""
    conf = specsynth.make_confidences()
    e = oracle.sched_exact(conf, COSTS["C"], 1)
    g = oracle.sched_alg1(conf, COSTS["C"], 1)
    assert e["verify_len"].sum() + 64 == 64 * 17
    assert g["verify_len"].sum() < e["verify_len"].sum()


# ------------------------------------------------------------- limit cases
def test_constant_cost_verifies_everything():
    conf = specsynth.make_confidences(16, 8, seed=7)
    r = oracle.sched_exact(conf, ([0.0], [5.0]), 0)
    assert (r["verify_len"] == 8).all()


def test_zero_survival_positions_are_not_verified_at_constant_cost():
    """Constant cost: positions with zero survival add nothing to tau, so the
    first (smallest-budget) maximum leaves them out."""
    conf = np.array([[0.9, 0.0, 0.5], [0.8, 0.7, 0.0]], np.float32)
    r = oracle.sched_exact(conf, ([0.0], [3.0]), 0)
    assert list(r["verify_len"]) == [1, 2]


def test_huge_slope_keeps_min_len():
    """C proportional to N: tau/N starts at 1 with anchors only and every
    survival is below 1, so nothing is added."""
    conf = specsynth.make_confidences(16, 8, seed=7)
    r = oracle.sched_exact(conf, ([0.0, 1e6], [1e-9, 1e15]), 0)
    assert (r["verify_len"] == 0).all()
    assert (oracle.sched_alg1(conf, ([0.0, 1e6], [1e-9, 1e15]), 0)["verify_len"] == 0).all()


def test_cost_cliff_keeps_min_len():
    """A cost that jumps by 1e9 right after the minimum budget keeps min_len."""
    conf = specsynth.make_confidences(16, 8, seed=7)
    for ml in (0, 1, 3):
        n0 = 16.0 * (ml + 1)
        r = oracle.sched_exact(conf, ([n0, n0 + 1.0], [1.0, 1e9]), ml)
        assert (r["verify_len"] == ml).all()


def test_contiguity_with_tied_survivals():
    """Confidences of exactly 1 make equal survivals inside a request; the
    shallow-first tie-break keeps every prefix contiguous (AngelSpec §4.2), so
    Algorithm 1 never meets a non-contiguous candidate and, under affine costs,
    still equals the count-based exact scan."""
    rng = np.random.default_rng(8)
    for trial in range(300):
        conf = rng.choice(np.array([1.0, 0.5, 0.25, 1.0, 0.75], np.float32), size=(6, 6))
        cost = ([0.0, 100.0], [float(rng.uniform(1, 30)), 100.0 + float(rng.uniform(1, 30))])
        e = oracle.sched_exact(conf, cost, 0)
        a = oracle.sched_alg1(conf, cost, 0)
        assert e["rc"] == 0 and a["rc"] == 0
        assert list(e["verify_len"]) == list(a["verify_len"])


def test_invalid_scheduler_inputs():
    conf = np.full((2, 3), 0.5, np.float32)
    assert oracle.sched_exact(conf, ([1.0, 1.0], [1.0, 2.0]))["rc"] == oracle.ERR_COST_TABLE
    assert oracle.sched_exact(conf, ([0.0, 1.0], [1.0, 0.0]))["rc"] == oracle.ERR_COST_TABLE
    bad = conf.copy()
    bad[1, 2] = 1.5
    assert oracle.sched_exact(bad, ([0.0], [1.0]))["rc"] == oracle.ERR_CONFIDENCE
    assert oracle.sched_exact(conf, ([0.0], [1.0]), 4)["rc"] == oracle.ERR_SHAPE


# ------------------------------------------- the choice, in exact arithmetic
def _exact_cost(N, cost):
    """C(N) of a knot table in exact rationals (knots taken as the doubles
    they are): linear between knots, flat beyond both ends."""
    from fractions import Fraction
    kt = [Fraction(float(t)) for t in cost[0]]
    kc = [Fraction(float(c)) for c in cost[1]]
    N = Fraction(N)
    if N <= kt[0]:
        return kc[0]
    if N >= kt[-1]:
        return kc[-1]
    i = max(j for j in range(len(kt) - 1) if kt[j] <= N)
    return kc[i] + (N - kt[i]) * (kc[i + 1] - kc[i]) / (kt[i + 1] - kt[i])


def _exact_argmax(conf, cost, min_len):
    """The allocation in [min_len, gamma]^B maximising tau / C(N) exactly:
    survivals s_{b,k} = prod_{t<k} c_{b,t} (AngelSpec eq. (20)) and progress
    A_b(l) = sum_{k<=l} s_{b,k} (eq. (21)) as exact rationals of the fp32
    confidences, tau = sum_b A_b(l_b), N = sum_b (l_b + 1) (eq. (24)).
    Returns (allocation, relative gap to the best other allocation)."""
    import itertools
    from fractions import Fraction
    B, gamma = conf.shape
    A = []
    for b in range(B):
        s, acc, row = Fraction(1), Fraction(1), [Fraction(1)]
        for k in range(gamma):
            s *= Fraction(float(conf[b, k]))
            acc += s
            row.append(acc)
        A.append(row)
    # every denominator is a power of two: integers over a common one
    D = max(a.denominator for row in A for a in row)
    Ai = [[a.numerator * (D // a.denominator) for a in row] for row in A]
    top = {}   # N -> two largest (tau, allocation)
    for alloc in itertools.product(range(min_len, gamma + 1), repeat=B):
        tau = sum(Ai[b][l] for b, l in enumerate(alloc))
        N = sum(alloc) + B
        best = top.setdefault(N, [])
        best.append((tau, alloc))
        best.sort(key=lambda t: -t[0])
        del best[2:]
    objs = []
    for N, best in top.items():
        C = _exact_cost(N, cost)
        for tau, alloc in best:
            objs.append((Fraction(tau, D) / C, alloc))
    objs.sort(key=lambda t: -t[0])
    gap = (objs[0][0] - objs[1][0]) / objs[0][0] if len(objs) > 1 else Fraction(1)
    return np.array(objs[0][1], np.int32), gap


def test_choice_with_survivals_closer_than_2_pow_minus_20():
    """Two candidates whose survivals differ by 4 fp32 ulps of 0.75 (2.4e-7):
    the exact order puts request 1 first, and a cost that stops after one
    extra position must extend request 1, not request 0."""
    c1 = np.float32(0.75) + np.float32(4 * 2.0 ** -24)
    conf = np.array([[0.75], [c1]], np.float32)
    cost = ([0.0, 3.0, 4.0], [1.0, 1.0, 100.0])
    alloc, gap = _exact_argmax(conf, cost, 0)
    assert list(alloc) == [0, 1] and gap > 1e-9
    assert list(oracle.sched_exact(conf, cost, 0)["verify_len"]) == [0, 1]


@pytest.mark.parametrize("cost_name", ["affine", "Bprime", "A", "C"])
@pytest.mark.parametrize("min_len", [0, 1])
def test_exact_scan_choice_is_the_exact_rational_argmax(cost_name, min_len):
    """The allocation the oracle's exact scan returns (fixed-point survivals,
    integer progress sums) is the argmax of tau / C over every allocation in
    exact rational arithmetic, whenever that argmax leads the next allocation
    by more than 1e-9 relative.  B <= 4, gamma <= 4; confidences uniform,
    sigmoid(N(1.5, 1)) as in the scheduled workload, or with near-tied
    survivals (a few fp32 ulps apart) planted between requests."""
    rng = np.random.default_rng(70 + min_len + 10 * ["affine", "Bprime", "A", "C"].index(cost_name))
    kt, kc = COSTS[cost_name]
    checked = 0
    trials = 2500
    for trial in range(trials):
        B = int(rng.integers(1, 5))
        gamma = int(rng.integers(max(1, min_len), 5))
        kind = trial % 3
        if kind == 0:
            conf = rng.uniform(0.0, 1.0, (B, gamma)).astype(np.float32)
        elif kind == 1:
            z = rng.normal(1.5, 1.0, (B, gamma))
            conf = (1.0 / (1.0 + np.exp(-z))).astype(np.float32)
        else:
            conf = rng.uniform(0.5, 1.0, (B, gamma)).astype(np.float32)
            for b in range(1, B):
                ulps = int(rng.integers(-6, 7))
                conf[b, 0] = np.float32(conf[0, 0] + np.float32(ulps * 2.0 ** -24))
        s = float(rng.uniform(0.002, 0.2))
        cost = (np.array(kt) * s, np.array(kc))
        if cost_name == "affine":
            cost = ([0.0, 10.0], [1.0, 1.0 + 10.0 * float(rng.uniform(0.01, 2.0))])
        r = oracle.sched_exact(conf, cost, min_len)
        assert r["rc"] == 0
        want, gap = _exact_argmax(conf, cost, min_len)
        if gap <= 1e-9:
            continue
        checked += 1
        assert np.array_equal(r["verify_len"], want), (trial, conf, r["verify_len"], want, float(gap))
    assert checked >= 0.9 * trials
