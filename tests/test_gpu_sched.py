"""Bit-exact parity of the CUDA scheduler with the oracle (exact scan and
Algorithm 1), through the C ABI."""
import numpy as np
import pytest

import oracle
import specsynth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_softmax_gb300 as m
    m.build()
    return m


def _gpu(sv, conf, cost, min_len, mode=0):
    import torch
    out, ws = sv.schedule(torch.from_numpy(np.ascontiguousarray(conf)).cuda(), cost, min_len, mode)
    st = sv.read_status(ws)
    return out.cpu().numpy(), st


@pytest.mark.parametrize("cost_name", ["Bprime", "A", "C", "affine"])
def test_scheduled_workload_cost_readings(sv, cost_name):
    conf = specsynth.make_confidences()
    cost = specsynth.COST_TABLES[cost_name]
    for mode, ref in ((0, oracle.sched_exact), (1, oracle.sched_alg1)):
        g, st = _gpu(sv, conf, cost, specsynth.SCHED_MIN_LEN, mode)
        assert st == 0
        assert (g == ref(conf, cost, specsynth.SCHED_MIN_LEN)["verify_len"]).all(), (cost_name, mode)


def test_random_draws_bit_exact(sv):
    rng = np.random.default_rng(77)
    for trial in range(400):
        B = int(rng.integers(1, 300))
        gamma = int(rng.integers(1, 33))
        ml = int(rng.integers(0, min(gamma, 3) + 1))
        if B * (gamma - ml) > 16384:
            continue
        conf = specsynth.make_confidences(B, gamma, seed=9000 + trial, mean=float(rng.uniform(-1, 3)))
        if trial % 7 == 0:
            conf[rng.random(conf.shape) < 0.2] = 1.0      # tied survivals
        if trial % 11 == 0:
            conf[rng.random(conf.shape) < 0.1] = 0.0      # zero survivals
        nk = int(rng.integers(1, 6))
        kt = np.cumsum(rng.uniform(1, B * (gamma + 1) / 2, nk))
        kc = rng.uniform(0.5, 30, nk)
        cost = (list(kt), list(kc))
        mode = trial % 2
        ref = (oracle.sched_exact if mode == 0 else oracle.sched_alg1)(conf, cost, ml)
        g, st = _gpu(sv, conf, cost, ml, mode)
        assert st == 0
        assert (g == ref["verify_len"]).all(), (trial, B, gamma, ml, mode)


def test_largest_candidate_count(sv):
    conf = specsynth.make_confidences(512, 32, seed=3)
    cost = specsynth.COST_TABLES["Bprime"]
    g, st = _gpu(sv, conf, cost, 0)
    assert st == 0 and (g == oracle.sched_exact(conf, cost, 0)["verify_len"]).all()
    conf = specsynth.make_confidences(4096, 4, seed=4)
    g, st = _gpu(sv, conf, ([0.0, 1e5], [4.0, 4.0 + 1e5 * 0.001]), 0)
    assert (g == oracle.sched_exact(conf, ([0.0, 1e5], [4.0, 4.0 + 1e5 * 0.001]), 0)["verify_len"]).all()


def test_min_len_equals_gamma(sv):
    conf = specsynth.make_confidences(8, 4, seed=5)
    g, st = _gpu(sv, conf, specsynth.COST_TABLES["A"], 4)
    assert (g == 4).all()


def test_invalid_confidence_sets_status(sv):
    conf = specsynth.make_confidences(8, 4, seed=5)
    conf[3, 2] = np.nan
    g, st = _gpu(sv, conf, specsynth.COST_TABLES["A"], 1)
    assert st == sv.ERR_CONFIDENCE and (g == -1).all()
