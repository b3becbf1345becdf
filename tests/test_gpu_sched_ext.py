"""Parity of the CUDA D-cut budget, static schedulers and STS-calibrated
schedules with the oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import specsynth

pytestmark = pytest.mark.gpu

RATIOS = [0.125, 0.25, 0.375, 0.5, 0.625, 0.75, 0.875, 1.0]


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_softmax_gb300 as m
    m.build()
    return m


def _dev(conf):
    import torch
    return torch.from_numpy(np.ascontiguousarray(conf, np.float32)).cuda()


def _dcut(sv, conf, costs, min_len=0, sts=None):
    out, ws = sv.schedule(_dev(conf), (RATIOS[:len(costs)], costs), min_len, sv.SCHED_DCUT, sts=sts)
    return out.cpu().numpy(), sv.read_status(ws)


def _costs(rng, n):
    """Verification cost rising with the budget (ms), like a batch latency curve."""
    return list(np.cumsum(rng.uniform(0.2, 2.0, n)) + rng.uniform(1.0, 10.0))


def test_dcut_bit_exact(sv):
    """Without calibration both sides do the same fp64 operations in the same
    order: allocations agree exactly, ties included (first maximum)."""
    rng = np.random.default_rng(31)
    for trial in range(300):
        B = int(rng.integers(1, 300))
        gamma = int(rng.integers(1, 33))
        ml = int(rng.integers(0, min(gamma, 3) + 1))
        if B * (gamma - ml) > 16384:
            continue
        conf = specsynth.make_confidences(B, gamma, seed=500 + trial, mean=float(rng.uniform(-1, 3)))
        if trial % 5 == 0:
            conf[rng.random(conf.shape) < 0.3] = 1.0
        nr = int(rng.integers(1, len(RATIOS) + 1))
        costs = _costs(rng, nr)
        ref = oracle.sched_dcut(conf, RATIOS[:nr], costs, ml)
        g, st = _dcut(sv, conf, costs, ml)
        assert st == 0 and ref["rc"] == 0
        assert (g == ref["verify_len"]).all(), (trial, B, gamma, ml, nr)


def test_dcut_exact_tie_takes_first_ratio(sv):
    conf = np.ones((4, 3), np.float32)
    g, st = _dcut(sv, conf, [4.0, 8.0, 12.0, 16.0])
    assert st == 0 and (g == 0).all()


def test_dcut_block_diffusion_shape(sv):
    """64 requests with 16 drafts each, the per-position confidence pattern of
    the block-diffusion workload."""
    conf = specsynth.make_confidences(64, 16, seed=11)
    costs = [6.0, 7.2, 8.3, 9.6, 10.5, 11.9, 13.0, 14.4]
    ref = oracle.sched_dcut(conf, RATIOS, costs)
    g, st = _dcut(sv, conf, costs)
    assert st == 0 and (g == ref["verify_len"]).all()


def _static(sv, conf, th, max_len, min_len=0, sts=None):
    out, ws = sv.schedule_static(_dev(conf), th, max_len, min_len, sts=sts)
    return out.cpu().numpy(), sv.read_status(ws)


def test_static_bit_exact(sv):
    rng = np.random.default_rng(41)
    for trial in range(200):
        B = int(rng.integers(1, 4097))
        gamma = int(rng.integers(1, 33))
        ml = int(rng.integers(0, gamma + 1))
        mx = int(rng.integers(ml, gamma + 1))
        conf = specsynth.make_confidences(B, gamma, seed=700 + trial, mean=float(rng.uniform(-1, 3)))
        # thresholds that are float32 values; some equal a confidence exactly
        th = float(np.float32(rng.uniform(0, 1))) if trial % 4 else float(conf.flat[int(rng.integers(conf.size))])
        if trial % 9 == 0:
            th = 0.0
        ref = oracle.sched_threshold(conf, th, ml, max_len=mx)
        g, st = _static(sv, conf, th, mx, ml)
        assert st == 0 and ref["rc"] == 0
        assert (g == ref["verify_len"]).all(), (trial, B, gamma, ml, mx, th)


def test_fixed_length(sv):
    conf = specsynth.make_confidences(128, 8, seed=2)
    g, st = _static(sv, conf, 0.0, 5)
    assert st == 0 and (g == 5).all()


def test_static_invalid_confidence_sets_status(sv):
    conf = specsynth.make_confidences(8, 4, seed=5)
    conf[2, 1] = 1.5
    g, st = _static(sv, conf, 0.5, 4)
    assert st == sv.ERR_CONFIDENCE and g[2] == -1
    ok = np.arange(8) != 2
    assert (g[ok] == oracle.sched_threshold(conf[ok], 0.5)["verify_len"]).all()
    # the status word is cleared by the next good call
    g, st = _static(sv, conf[ok], 0.5, 4)
    assert st == 0


# -------------------------------------------------------------- STS inputs
def _sts(rng, gamma):
    """Temperatures on the fit's grid, as the float32 values the library takes."""
    return ((rng.integers(1, 101, gamma)) / 10.0).astype(np.float32)


def _calibrated(conf, T):
    return conf.astype(np.float64) ** (1.0 / T.astype(np.float64))[None, :]


def test_sts_threshold(sv):
    """Device and host pow may differ in the last bits, so a calibrated
    confidence within 1e-12 of the threshold may fall either way: such
    requests are compared up to the first near-tie only."""
    rng = np.random.default_rng(51)
    requests = excused = 0
    for trial in range(60):
        B = int(rng.integers(1, 2000))
        gamma = int(rng.integers(1, 33))
        conf = specsynth.make_confidences(B, gamma, seed=900 + trial, mean=float(rng.uniform(-1, 3)))
        T = _sts(rng, gamma)
        th = float(np.float32(rng.uniform(0.05, 0.95)))
        ref = oracle.sched_threshold(conf, th, 0, sts_T=T.astype(np.float64))["verify_len"]
        g, st = _static(sv, conf, th, gamma, 0, sts=T)
        assert st == 0
        near = np.abs(_calibrated(conf, T) - th) < 1e-12
        first_near = np.where(near.any(axis=1), near.argmax(axis=1), gamma + 1)
        clear = ref < first_near
        assert (g[clear] == ref[clear]).all()
        assert (np.minimum(g, first_near) == np.minimum(ref, first_near)).all()
        requests += B
        excused += int((~clear & (g != ref)).sum())
    print(f"\n[sts threshold] requests={requests} excused near-ties={excused}")
    assert excused <= 1e-3 * requests


def test_sts_unit_temperatures_change_nothing(sv):
    conf = specsynth.make_confidences(256, 8, seed=3)
    cost = specsynth.COST_TABLES["Bprime"]
    ones = np.ones(8, np.float32)
    a, ws = sv.schedule(_dev(conf), cost, 1, sv.SCHED_EXACT, sts=ones)
    b, _ = sv.schedule(_dev(conf), cost, 1, sv.SCHED_EXACT)
    assert sv.read_status(ws) == 0 and (a.cpu() == b.cpu()).all()


@pytest.mark.parametrize("mode", ["exact", "alg1", "dcut"])
def test_sts_schedules(sv, mode):
    """Calibrated survivals are products of pow(); trials whose optimum is
    within 1e-9 (relative) of another allocation's objective are skipped,
    every other trial must agree exactly."""
    rng = np.random.default_rng({"exact": 61, "alg1": 62, "dcut": 63}[mode])
    checked = excused = 0
    for trial in range(80):
        B = int(rng.integers(1, 200))
        gamma = int(rng.integers(1, 33))
        if B * gamma > 16384:
            continue
        conf = specsynth.make_confidences(B, gamma, seed=1100 + trial, mean=float(rng.uniform(-1, 3)))
        T = _sts(rng, gamma)
        T64 = T.astype(np.float64)
        if mode == "dcut":
            costs = _costs(rng, len(RATIOS))
            ref = oracle.sched_dcut(conf, RATIOS, costs, 0, sts_T=T64)
            o = np.sort(ref["obj"])
            if o[-1] - o[-2] < 1e-9 * o[-1]:
                continue
            g, st = _dcut(sv, conf, costs, 0, sts=T)
        else:
            cost = specsynth.COST_TABLES["Bprime"]
            ex = oracle.sched_exact(conf, cost, 0, sts_T=T64)
            if ex["gap"] < 1e-9:
                continue
            ref = ex if mode == "exact" else oracle.sched_alg1(conf, cost, 0, sts_T=T64)
            out, ws = sv.schedule(_dev(conf), cost, 0, sv.SCHED_EXACT if mode == "exact" else sv.SCHED_ALGORITHM1,
                                  sts=T)
            g, st = out.cpu().numpy(), sv.read_status(ws)
        assert st == 0
        # an allocation is fixed by its count of candidates; candidates with
        # calibrated survivals within rounding of each other may swap
        s = np.cumprod(_calibrated(conf, T), axis=1)
        if not (g == ref["verify_len"]).all():
            assert g.sum() == ref["verify_len"].sum()
            prog = lambda v: sum(s[b, :v[b]].sum() for b in range(B))
            assert abs(prog(g) - prog(ref["verify_len"])) <= 1e-12 * prog(ref["verify_len"]), trial
            excused += 1
        checked += 1
    print(f"\n[sts {mode}] trials checked={checked} excused (equal count and progress)={excused}")
    assert checked > 40
    assert excused <= max(1, 0.05 * checked)


def test_sts_fit_from_verify_outcomes(sv):
    """The calibration loop: verify every draft position of a batch, take each
    draft's own probability q(x) as its confidence, fit STS temperatures on
    the observed accept lengths, and schedule with them."""
    import torch
    case = specsynth.make_verify_case("tiny", B=2048, V=64, seed_logits=610, seed_noise=611, seed_tokens=612,
                                      seed_uniforms=613)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out_t, out_n, ws = sv.verify(dev(case.target), dev(case.draft), dev(case.draft_tokens), dev(case.verify_len),
                                 case.T, dev(case.uniforms))
    al = out_n.cpu().numpy()
    ref = oracle.verify(case.target, case.draft, case.dtype, case.draft_tokens, case.verify_len, case.T,
                        case.uniforms)
    assert (al == ref["accept_len"]).sum() >= al.size - 1      # near-ties may differ, none seen so far
    _, qx, _, st = sv.verify_stats(ws, case.B, case.gamma, case.V, sv.F32)
    assert (st.cpu().numpy() == 0).all()
    conf = qx.cpu().numpy().astype(np.float32)
    T, e = sv.sts_fit(conf, al)
    r = oracle.sts_fit(conf, al)
    np.testing.assert_array_equal(T, r["T"].astype(np.float32))
    # the fit never does worse than leaving position 1 uncalibrated (T = 1 is on the grid)
    assert e[0] <= oracle.sts_ece(conf[:, 0].astype(np.float64), (al >= 1).astype(np.int32)) + 1e-15
    g, st2 = _static(sv, conf, 0.5, case.gamma, 0, sts=T)
    assert st2 == 0
    want = oracle.sched_threshold(conf, 0.5, 0, sts_T=T.astype(np.float64))["verify_len"]
    near = (np.abs(_calibrated(conf, T) - 0.5) < 1e-12).any(axis=1)
    assert (g[~near] == want[~near]).all()
