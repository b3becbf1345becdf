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


@pytest.mark.parametrize("name,T", [("mtp_chat", None), ("greedy", 0.0)])
def test_streaming_kernel_timeout_path(sv, name, T):
    """The real streaming kernel's timeout path: with the test hook on, the
    first copy wait of every warp counts as expired; the warps let their
    copies land and stop, the call reports SPEC_ERR_TIMEOUT and marks every
    request invalid.  The next call on the same workspace, hook off, matches
    the oracle."""
    import numpy as np
    case = specsynth.make_verify_case(name, B=8, V=20000)
    T = case.T if T is None else T
    t, d, x, vl, u = specsynth.to_device(case)
    uu = u if T != 0 else None
    sv.selftest_expire_first_wait(True)
    try:
        tok, n, ws = sv.verify(t, d, x, vl, T, uu)
        st = sv.read_status(ws)
    finally:
        sv.selftest_expire_first_wait(False)
    assert st == sv.ERR_TIMEOUT
    assert (n.cpu().numpy() == -1).all() and (tok.cpu().numpy() == -1).all()
    tok, n, ws = sv.verify(t, d, x, vl, T, uu, workspace=ws)
    assert sv.read_status(ws) == 0
    o = H.oracle_verify(case, T=T)
    P = H.compare(o, tok.cpu().numpy(), n.cpu().numpy(), greedy=T == 0)
    H.assert_parity(P, prob=False)
    assert (n.cpu().numpy() >= 0).all()
