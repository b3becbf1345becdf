"""spec_verify_static, the workspace-free entry point, agrees with spec_verify.

It exists for callers that cannot allocate device memory where they verify;
its scratch is a fixed array in device memory shared by all calls.  Two calls
in a row (different shapes, so the second runs over the first one's leftovers)
must give exactly the outputs of spec_verify on the same inputs.  This file is
collected last and also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import specsynth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_softmax_gb300 as m
    m.build()
    return m


def _both(sv, case, T=None):
    T = case.T if T is None else T
    t, d, x, vl, u = H.to_device(case)
    uu = u if T != 0 else None
    ref_tok, ref_n, _ = sv.verify(t, d, x, vl, T, uu)
    tok, n = sv.verify_static(t, d, x, vl, T, uu)
    return ref_tok.cpu().numpy(), ref_n.cpu().numpy(), tok.cpu().numpy(), n.cpu().numpy()


def test_two_calls_in_a_row_match_spec_verify(sv):
    first = specsynth.make_verify_case("mtp_chat")                   # B=16, V=32000, T=0.8
    second = specsynth.make_verify_case("block_diffusion", B=24)     # larger scratch footprint
    for case in (first, second):
        rt, rn, st, sn = _both(sv, case)
        assert np.array_equal(rn, sn)
        assert np.array_equal(rt, st)
        assert (sn >= 0).all()


def test_greedy_and_invalid_requests(sv):
    case = specsynth.make_verify_case("tiny", B=6)
    case.draft_tokens[2, 0] = case.V                # invalid token -> marked per request
    rt, rn, st, sn = _both(sv, case)
    assert np.array_equal(rn, sn) and np.array_equal(rt, st)
    assert sn[2] == -1
    g = specsynth.make_verify_case("greedy", B=4, V=3001)
    rt, rn, st, sn = _both(sv, g)
    assert np.array_equal(rn, sn) and np.array_equal(rt, st)


def test_rejects_sizes_beyond_the_static_scratch(sv):
    need = sv.verify_workspace_bytes(4096, 32, 151936, sv.BF16)
    assert need > sv.STATIC_WORKSPACE_BYTES
    fake = ctypes.c_void_p(0x10000)
    rc = sv.lib().spec_verify_static(fake, fake, sv.BF16, 4096, 32, 151936, fake, None, ctypes.c_float(1.0),
                                     fake, fake, fake, None)
    assert rc == sv.ERR_WORKSPACE
