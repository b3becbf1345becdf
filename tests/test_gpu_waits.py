"""The bounded waits end: a wait on a barrier that nothing completes gives up
after its limit and reports a timeout, the context stays usable, and a normal
verification call afterwards still matches the oracle."""
import pytest

import specsynth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_softmax_gb300 as m
    m.build()
    return m


@pytest.mark.parametrize("limit_ns", [1_000_000, 20_000_000])
def test_wait_gives_up_after_its_limit(sv, limit_ns):
    (st_blocked, st_done), (el_blocked, el_done) = sv.selftest_wait(limit_ns)
    assert st_blocked == sv.ERR_TIMEOUT
    assert limit_ns <= el_blocked < limit_ns + 50_000_000
    assert st_done == sv.OK and el_done < 1_000_000


def test_context_usable_after_a_timeout(sv):
    sv.selftest_wait(1_000_000)
    case = specsynth.make_verify_case("tiny")
    g = H.gpu_verify(case)
    o = H.oracle_verify(case)
    P = H.compare(o, g["tokens"], g["accept_len"], g["px"], g["qx"], g["mass"], g["status"])
    assert g["device_status"] == 0
    H.assert_parity(P)
