"""The library's host STS fit (spec_sts_fit) against the oracle's fit.  Host
code only: no GPU is touched."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_softmax_gb300 as m
    m.build()
    return m


def _case(seed, n, gamma, power):
    rng = np.random.default_rng(seed)
    conf = (1 / (1 + np.exp(-rng.normal(1.0, 1.2, (n, gamma))))).astype(np.float32)
    acc = rng.random((n, gamma)) < conf.astype(np.float64) ** power
    al = np.where(~acc, np.arange(gamma)[None, :], gamma).min(axis=1).astype(np.int32)
    return conf, al


@pytest.mark.parametrize("seed,n,gamma,power", [(1, 3000, 4, 1.0), (2, 5000, 8, 2.0), (3, 2000, 16, 0.6),
                                                (4, 1, 1, 1.0), (5, 37, 32, 1.5)])
def test_library_fit_matches_oracle(sv, seed, n, gamma, power):
    conf, al = _case(seed, n, gamma, power)
    T, e = sv.sts_fit(conf, al)
    ref = oracle.sts_fit(conf, al)
    assert ref["rc"] == 0
    np.testing.assert_array_equal(T, ref["T"].astype(np.float32))
    np.testing.assert_allclose(e, ref["ece"], rtol=0, atol=1e-15)


def test_fit_rejects_bad_input(sv):
    conf, al = _case(1, 10, 4, 1.0)
    bad = conf.copy()
    bad[3, 1] = np.nan
    with pytest.raises(RuntimeError):
        sv.sts_fit(bad, al)
    with pytest.raises(RuntimeError):
        sv.sts_fit(np.zeros((4, 33), np.float32), np.zeros(4, np.int32))
