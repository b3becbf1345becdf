"""The parity harness itself: a wrong GPU answer must not pass.

The GPU side is simulated on the CPU by copying the oracle's own outputs and
planting mistakes in them (a drawn token one bin or a few bins off, a token far
away, a shortened accepted prefix).  The comparison excuses a different drawn
token only where the draw's uniform lies within 1e-5 of the oracle's own bin
of that token; every other planted mistake must be reported.
"""
import numpy as np
import pytest

import specsynth
from tests import _helpers as H


@pytest.fixture(scope="module")
def block_diffusion():
    case = specsynth.make_verify_case("block_diffusion")
    return case, H.oracle_verify(case)


def _emitted(o):
    n = o["accept_len"]
    return n, o["tokens"][np.arange(len(n)), n]


def test_identical_outputs_pass(block_diffusion):
    case, o = block_diffusion
    P = H.compare(o, o["tokens"].copy(), o["accept_len"].copy())
    H.assert_parity(P, prob=False)
    assert P.positions == int((o["accept_len"] + 1).sum()) and P.flagged == 0


@pytest.mark.parametrize("shift", [1, -1, 3])
def test_draw_a_few_bins_off_is_rejected(block_diffusion, shift):
    """Every drawn token moved by `shift`: excused only where u is within 1e-5
    (normalised CDF) of the boundary towards the planted token, checked here
    from the oracle's own edges of its drawn bin; the bar then fails."""
    case, o = block_diffusion
    n, tok = _emitted(o)
    g = o["tokens"].copy()
    planted = np.clip(tok + shift, 0, case.V - 1)
    moved = planted != tok
    g[np.arange(case.B), n] = planted
    P = H.compare(o, g, o["accept_len"].copy())
    assert len(P.mismatches) + P.draw_flagged == int(moved.sum())
    excused = {b for b in range(case.B) if moved[b]} - {m[0] for m in P.mismatches}
    for b in excused:
        # the planted bin starts (or ends) where the oracle's bin ends (or
        # starts) up to empty bins in between; u must be that close to it
        lo, hi = o["cdf_lo"][b], o["cdf_hi"][b]
        gap = (hi - o["u_draw"][b]) if shift > 0 else (o["u_draw"][b] - lo)
        assert gap < H.DRAW_FLAG, (b, gap)
    assert len(P.mismatches) > case.B // 2
    with pytest.raises(AssertionError):
        H.assert_parity(P, prob=False)


def test_far_token_near_an_edge_is_rejected(block_diffusion):
    """Where u lies within 1e-5 of an edge of the oracle's bin, a token on the
    far side of the vocabulary is still a mismatch (an excuse that looked only
    at the oracle's bin would let it through)."""
    case, o = block_diffusion
    n, tok = _emitted(o)
    near = np.minimum(o["u_draw"] - o["cdf_lo"], o["cdf_hi"] - o["u_draw"]) < H.DRAW_FLAG
    assert near.sum() >= 4   # at this vocabulary size many draws sit that close to an edge
    g = o["tokens"].copy()
    g[np.arange(case.B), n] = np.where(near, (tok + case.V // 2) % case.V, tok)
    P = H.compare(o, g, o["accept_len"].copy())
    assert {m[0] for m in P.mismatches} == set(np.flatnonzero(near).tolist())
    assert P.draw_flagged == 0


def test_shortened_prefix_is_rejected(block_diffusion):
    """An accepted prefix one shorter is excused only at an accept near-tie
    (|u - p/q| < 1e-5), which none of these positions is."""
    case, o = block_diffusion
    n, tok = _emitted(o)
    g_len = o["accept_len"].copy()
    g_tok = o["tokens"].copy()
    hit = np.flatnonzero(n > 0)
    g_len[hit] -= 1
    P = H.compare(o, g_tok, g_len)
    assert {m[0] for m in P.mismatches} == set(hit.tolist())


def test_flag_budget():
    """Flagged positions are held below 1e-4 of the positions."""
    P = H.Parity(positions=20000, accept_flagged=1, draw_flagged=1)
    H.assert_parity(P, prob=False)
    P = H.Parity(positions=20000, accept_flagged=2, draw_flagged=1)
    with pytest.raises(AssertionError):
        H.assert_parity(P, prob=False)
