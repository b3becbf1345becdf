"""Pins of the verification oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the worked
example's printed numbers, exact enumeration of the accept/resample process,
chi-square and binomial tests against the target distribution, the
expected-accepted-length closed form, and special cases that reduce to plain
sampling or greedy argmax.
"""
import json
import os

import numpy as np
import pytest
from scipy import stats

import oracle
import specsynth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _worked():
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        return json.load(f)


def _probs_case(p_rows, q_rows, x, u):
    P = np.array([p_rows], np.float64)
    Q = np.array([q_rows], np.float64)
    return oracle.verify_probs(P, Q, np.array([x], np.int32), np.array([u], np.float64))


# --------------------------------------------------------------- worked example
def test_worked_example_accept_boundary():
    """Token 1 has p/q = 0.3/0.5 = 0.6: accepted for u just below, rejected above."""
    g = _worked()
    p, q = g["p_target"], g["q_draft"]
    # gamma = 1: slots [accept_0, residual, bonus]
    acc = _probs_case([p, p], [q], [1], [0.59, 0.5, 0.5])
    rej = _probs_case([p, p], [q], [1], [0.61, 0.5, 0.5])
    assert acc["accept_len"][0] == 1 and acc["tokens"][0, 0] == 1
    assert rej["accept_len"][0] == 0


@pytest.mark.parametrize("x", [0, 2])
def test_worked_example_always_accept_where_p_ge_q(x):
    g = _worked()
    p, q = g["p_target"], g["q_draft"]
    for u in (0.0, 0.5, 0.999999):
        r = _probs_case([p, p], [q], [x], [u, 0.5, 0.5])
        assert r["accept_len"][0] == 1 and r["tokens"][0, 0] == x


def test_worked_example_residual_mass_and_draws():
    """Residual = [0.1, 0, 0.1], mass 0.2 = 1 - overlap; normalised [0.5, 0, 0.5]:
    u = 0.49 -> token 0, u = 0.51 -> token 2, and the zero bin 1 is never drawn."""
    g = _worked()
    p, q = g["p_target"], g["q_draft"]
    r49 = _probs_case([p, p], [q], [1], [0.99, 0.49, 0.5])
    r51 = _probs_case([p, p], [q], [1], [0.99, 0.51, 0.5])
    assert r49["accept_len"][0] == 0 and r49["tokens"][0, 0] == 0
    assert r51["accept_len"][0] == 0 and r51["tokens"][0, 0] == 2
    assert abs(r49["resid_mass"][0] - g["p_sticks_up_sum"]) < 1e-12
    assert abs(r49["resid_mass"][0] - (1.0 - g["overlap_sum"])) < 1e-12
    # residual draw never lands in the zero-weight bin, whatever u
    edge = g["residual_normalised"][0]
    for u in ((np.arange(2000) + 0.5) / 2000)[::37]:
        r = _probs_case([p, p], [q], [1], [0.99, u, 0.5])
        assert r["tokens"][0, 0] == (0 if u < edge else 2)


def test_draw_skips_leading_zero_weight_bins():
    """Residual [0, 0.1, 0.1]: even u = 0 must not draw the empty bin 0 (the CDF
    test is strict)."""
    p, q = [0.3, 0.5, 0.2], [0.5, 0.4, 0.1]
    r = _probs_case([p, p], [q], [0], [0.99, 0.0, 0.5])
    assert r["accept_len"][0] == 0 and r["tokens"][0, 0] == 1


def test_worked_example_emitted_distribution_equals_p():
    """Exact enumeration over x ~ q and a fine grid of u: P(emit v) = p(v)."""
    g = _worked()
    p, q = np.array(g["p_target"]), np.array(g["q_draft"])
    n, m = 2000, 50
    ua = (np.arange(n) + 0.5) / n          # accept uniform grid
    ur = (np.arange(m) + 0.5) / m          # residual uniform grid (independent)
    B = 3 * n * m
    P = np.broadcast_to(np.array([p, p]), (B, 2, 3))
    Q = np.broadcast_to(np.array([q]), (B, 1, 3))
    X, IA, IR = np.meshgrid(np.arange(3), np.arange(n), np.arange(m), indexing="ij")
    xs, ia, ir = X.ravel(), IA.ravel(), IR.ravel()
    us = np.stack([ua[ia], ur[ir], np.full(B, 0.5)], axis=1)
    ws = q[xs] / (n * m)
    out = oracle.verify_probs(P, Q, xs.astype(np.int32)[:, None], us)
    emitted = out["tokens"][:, 0]
    dist = np.zeros(3)
    np.add.at(dist, emitted, ws)
    np.testing.assert_allclose(dist, p, atol=1e-9)
    # acceptance probability of the step equals the overlap 0.8
    acc = np.sum(ws[out["accept_len"] == 1])
    assert abs(acc - g["overlap_sum"]) < 1e-9


def test_worked_example_through_logits():
    """Same decisions when p, q enter as fp32 log-probability logits at T = 1."""
    g = _worked()
    p, q = np.array(g["p_target"]), np.array(g["q_draft"])
    c = specsynth.make_replicated_case(np.array([p, p]), np.array([q]), 4, 11, 12)
    c.draft_tokens[:] = 1
    c.uniforms[:] = np.array([[0.59, 0.5, 0.5], [0.61, 0.49, 0.5], [0.61, 0.51, 0.5],
                              [0.2, 0.5, 0.5]], np.float32)
    r = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, c.T, c.uniforms)
    assert list(r["accept_len"]) == [1, 0, 0, 1]
    assert list(r["tokens"][:, 0]) == [1, 0, 2, 1]
    np.testing.assert_allclose(r["px"][:, 0], 0.3, atol=1e-7)
    np.testing.assert_allclose(r["qx"][:, 0], 0.5, atol=1e-7)
    np.testing.assert_allclose(r["resid_mass"][1:3], 0.2, atol=1e-7)


def test_draw_cdf_edges_of_the_worked_example():
    """The oracle's CDF lookup on the page's example: after the rejection of
    token 1 the normalised residual is [0.5, 0, 0.5], so the bins are [0, .5),
    the empty [.5, .5) and [.5, 1); after acceptance the bonus draw uses p =
    [.5, .3, .2], bins [0, .5), [.5, .8), [.8, 1).  fp32 logits: 1e-6."""
    g = _worked()
    p, q = np.array(g["p_target"]), np.array(g["q_draft"])
    c = specsynth.make_replicated_case(np.array([p, p]), np.array([q]), 2, 11, 12)
    c.draft_tokens[:] = 1
    c.uniforms[:] = np.array([[0.61, 0.49, 0.5], [0.2, 0.5, 0.5]], np.float32)
    r = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, c.T, c.uniforms)
    assert list(r["accept_len"]) == [0, 1]
    res = np.cumsum([0.0] + g["residual_normalised"])
    lo, hi = oracle.draw_cdf(c.target, c.draft, c.dtype, c.verify_len, c.T, 0, 0, [0, 1, 2])
    np.testing.assert_allclose(lo, res[:3], atol=1e-6)
    np.testing.assert_allclose(hi, res[1:], atol=1e-6)
    cp = np.cumsum([0.0] + g["p_target"])
    lo, hi = oracle.draw_cdf(c.target, c.draft, c.dtype, c.verify_len, c.T, 1, 1, [0, 1, 2])
    np.testing.assert_allclose(lo, cp[:3], atol=1e-6)
    np.testing.assert_allclose(hi, cp[1:], atol=1e-6)


@pytest.mark.parametrize("name", ["tiny", "mtp_chat"])
def test_draw_cdf_brackets_the_drawn_token(name):
    """For every request the lookup gives the drawn token's bin exactly as the
    draw reported it, u lies inside it, and the bins of all tokens tile [0, 1]
    in order (hi of v = lo of v + 1, from 0 to 1)."""
    c = specsynth.make_verify_case(name, B=8, V=3000)
    r = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, c.T, c.uniforms)
    for b in range(c.B):
        n = int(r["accept_len"][b])
        tok = int(r["tokens"][b, n])
        lo, hi = oracle.draw_cdf(c.target, c.draft, c.dtype, c.verify_len, c.T, b, n, np.arange(c.V))
        assert lo[tok] == r["cdf_lo"][b] and hi[tok] == r["cdf_hi"][b]
        assert lo[tok] <= r["u_draw"][b] < hi[tok]
        assert lo[0] == 0.0 and abs(hi[-1] - 1.0) < 1e-15
        assert (hi[:-1] == lo[1:]).all() and (hi >= lo).all()


# ------------------------------------------------------------------ statistics
def _softmax64(z, T):
    """softmax(z / T) in fp64, with T the fp32 temperature widened."""
    y = z.astype(np.float64) / float(np.float32(T))
    e = np.exp(y - y.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,V", [(0.6, 7), (1.0, 300), (1.7, 2049)])
def test_logit_path_against_overlap_identity(dtype, T, V):
    """Through the logit path: p(x) and q(x) agree with a softmax computed here
    in fp64; the accept decisions are the first u * q(x) >= p(x); at a rejection
    the residual mass is sum max(p - q, 0) = 1 - sum min(p, q) (total variation,
    AngelSpec eqs. (4)-(5)); after full acceptance the bonus weights sum to 1.
    All to 1e-12."""
    rng = np.random.default_rng(int(V * 10 + T * 10) + (dtype == "bf16"))
    B, gamma = 96, 3
    zt32 = rng.normal(0.0, 2.0, (B, gamma + 1, V)).astype(np.float32)
    zd32 = (zt32[:, :gamma] + rng.normal(0.0, 1.0, (B, gamma, V))).astype(np.float32)
    if dtype == "bf16":
        zt, zd = specsynth.to_bf16_bits(zt32), specsynth.to_bf16_bits(zd32)
        zt32, zd32 = specsynth.bf16_bits_to_f32(zt), specsynth.bf16_bits_to_f32(zd)
    else:
        zt, zd = zt32, zd32
    P, Q = _softmax64(zt32, T), _softmax64(zd32, T)
    x = np.array([[rng.choice(V, p=Q[b, j]) for j in range(gamma)] for b in range(B)], np.int32)
    u = rng.uniform(0.0, 1.0, (B, gamma + 2)).astype(np.float32)
    r = oracle.verify(zt, zd, dtype, x, None, T, u)
    assert r["rc"] == 0 and (r["status"] == 0).all()
    n = r["accept_len"]
    rejected = 0
    for b in range(B):
        px = P[b, np.arange(gamma), x[b]]
        qx = Q[b, np.arange(gamma), x[b]]
        assert np.allclose(r["px"][b], px, rtol=1e-12, atol=0)
        assert np.allclose(r["qx"][b], qx, rtol=1e-12, atol=0)
        lhs = u[b, :gamma].astype(np.float64) * qx
        assert np.abs(lhs - px).min() > 1e-12 * px.max()  # no near-tie in these draws
        rej = np.flatnonzero(lhs >= px)
        want = int(rej[0]) if rej.size else gamma
        assert n[b] == want
        if want < gamma:
            rejected += 1
            tv = np.maximum(P[b, want] - Q[b, want], 0.0).sum()
            assert abs(r["resid_mass"][b] - tv) < 1e-12
            assert abs(r["resid_mass"][b] - (1.0 - np.minimum(P[b, want], Q[b, want]).sum())) < 1e-12
        else:
            assert abs(r["resid_mass"][b] - 1.0) < 1e-12
    assert 0 < rejected < B


def _dirichlet_rows(rng, rows, V, conc=1.0):
    return rng.dirichlet(np.full(V, conc), size=rows)


@pytest.fixture(scope="module")
def chi_case():
    rng = np.random.default_rng(2024)
    gamma, V, B = 3, 5, 1_000_000
    P = _dirichlet_rows(rng, gamma + 1, V)
    Q = _dirichlet_rows(rng, gamma, V)
    c = specsynth.make_replicated_case(P, Q, B, seed_tokens=71, seed_uniforms=72)
    r = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, c.T, c.uniforms)
    return P, Q, c, r


def _chi2_p(counts, probs):
    counts = np.asarray(counts, np.float64)
    exp = probs * counts.sum()
    return stats.chisquare(counts, exp).pvalue


@pytest.mark.slow
def test_chisquare_first_token_is_p0(chi_case):
    P, Q, c, r = chi_case
    first = r["tokens"][:, 0]
    assert _chi2_p(np.bincount(first, minlength=P.shape[1]), P[0]) > 1e-4


@pytest.mark.slow
def test_chisquare_second_token_given_first_accepted_is_p1(chi_case):
    P, Q, c, r = chi_case
    sel = r["accept_len"] >= 1
    second = r["tokens"][sel, 1]
    assert _chi2_p(np.bincount(second, minlength=P.shape[1]), P[1]) > 1e-4


@pytest.mark.slow
def test_chisquare_bonus_is_p_gamma(chi_case):
    P, Q, c, r = chi_case
    g = Q.shape[0]
    sel = r["accept_len"] == g
    bonus = r["tokens"][sel, g]
    assert sel.sum() > 10000
    assert _chi2_p(np.bincount(bonus, minlength=P.shape[1]), P[g]) > 1e-4


@pytest.mark.slow
def test_acceptance_rate_and_expected_length_closed_form(chi_case):
    """Per-position acceptance = overlap alpha_j = sum min(p_j, q_j) (AngelSpec eq. 5),
    and E[accepted] = sum_j prod_{i<=j} alpha_i (UraionSpec eq. expected_tau minus the
    bonus), each within 4 sigma."""
    P, Q, c, r = chi_case
    g = Q.shape[0]
    alpha = np.minimum(P[:g], Q).sum(axis=1)
    n = r["accept_len"]
    for j in range(g):
        reached = n >= j
        acc = (n[reached] > j).mean()
        sigma = np.sqrt(alpha[j] * (1 - alpha[j]) / reached.sum())
        assert abs(acc - alpha[j]) < 4 * sigma, (j, acc, alpha[j])
    expect = sum(np.prod(alpha[: j + 1]) for j in range(g))
    sigma = n.std() / np.sqrt(n.size)
    assert abs(n.mean() - expect) < 4 * sigma


@pytest.mark.slow
def test_residual_mass_is_one_minus_acceptance(chi_case):
    """The oracle's residual mass at the rejected row equals one minus the
    empirical acceptance rate of that row (TV = 1 - overlap, AngelSpec eqs. 4-5):
    two separate parts of the oracle agree."""
    P, Q, c, r = chi_case
    n = r["accept_len"]
    rejected0 = n == 0
    mass = r["resid_mass"][rejected0]
    assert np.allclose(mass, mass[0], atol=1e-12)
    acc0 = 1.0 - rejected0.mean()
    sigma = np.sqrt(acc0 * (1 - acc0) / n.size)
    assert abs((1.0 - mass[0]) - acc0) < 4 * sigma


# -------------------------------------------------------------- special cases
def test_equal_distributions_accept_everything():
    c = specsynth.make_verify_case("tiny", B=8)
    c.draft[:] = c.target[:, :-1]
    c.draft_tokens[:] = specsynth.gumbel_argmax(
        c.draft.reshape(-1, c.V), 1.0, 99).reshape(c.B, c.gamma)
    r = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, c.T, c.uniforms)
    assert (r["accept_len"] == c.gamma).all()
    assert (r["tokens"][:, : c.gamma] == c.draft_tokens).all()


def test_zero_length_is_a_plain_draw_from_p():
    rng = np.random.default_rng(5)
    V, B = 6, 400_000
    p = rng.dirichlet(np.ones(V))
    c = specsynth.make_replicated_case(np.array([p, p]), np.array([p]), B, 3, 4, verify_len=0)
    r = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, c.T, c.uniforms)
    assert (r["accept_len"] == 0).all()
    assert (r["tokens"][:, 1] == -1).all()
    assert _chi2_p(np.bincount(r["tokens"][:, 0], minlength=V), p) > 1e-4
    # ell = 0 uses the bonus slot gamma + 1: the inverse CDF of p at that uniform
    cdf = np.cumsum(p)
    u = c.uniforms[:1000, 2].astype(np.float64)
    expect = np.searchsorted(cdf, u, side="right")
    assert (r["tokens"][:1000, 0] == expect).all()


def test_one_hot_target_is_deterministic():
    V = 16
    c = specsynth.make_verify_case("tiny", B=6, V=V)
    c.target[:] = -1e4
    c.target[:, :, 7] = 0.0
    c.draft[:] = 0.0
    c.draft_tokens[:] = 3
    r = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, c.T, c.uniforms)
    assert (r["accept_len"] == 0).all()
    assert (r["tokens"][:, 0] == 7).all()


def test_single_token_vocabulary():
    c = specsynth.make_verify_case("tiny", B=3, V=1)
    c.draft_tokens[:] = 0
    r = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, c.T, c.uniforms)
    assert (r["accept_len"] == c.gamma).all()
    assert (r["tokens"] == 0).all()


def test_small_temperature_matches_greedy():
    """Top-1 margin >= 0.1 and T = 1e-3: the sampling path gives the greedy result."""
    c = specsynth.make_verify_case("tiny", B=16, V=64)
    tf = specsynth.as_f32(c.target, c.dtype)
    # enforce a top-1 margin of at least 0.1 in every target row
    am = tf.argmax(-1)
    srt = np.sort(tf, axis=-1)
    gap = srt[..., -1] - srt[..., -2]
    bump = np.maximum(0.0, 0.1 - gap) + 0.01
    for b in range(c.B):
        for j in range(c.gamma + 1):
            c.target[b, j, am[b, j]] += np.float32(bump[b, j])
    tf = specsynth.as_f32(c.target, c.dtype)
    greedy = tf.argmax(-1).astype(np.int32)
    rng = np.random.default_rng(1)
    c.draft_tokens[:] = np.where(rng.random((c.B, c.gamma)) < 0.8, greedy[:, :-1],
                                 rng.integers(0, 64, (c.B, c.gamma)))
    c.draft[:] = c.target[:, :-1]          # the draft agrees with the target
    c.uniforms[:] = np.minimum(c.uniforms, np.float32(1 - 1e-6))
    rg = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, 0.0, None)
    rs = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, 1e-3, c.uniforms)
    assert (rg["accept_len"] == rs["accept_len"]).all()
    assert (rg["tokens"] == rs["tokens"]).all()


def test_greedy_rule_by_hand():
    c = specsynth.make_verify_case("tiny", B=1, V=8, gamma=3)
    c.target[:] = 0.0
    c.target[0, 0, 2] = 1.0
    c.target[0, 1, 5] = 1.0
    c.target[0, 2, 1] = 1.0
    c.target[0, 3, 4] = 1.0
    c.target[0, 2, 6] = 1.0          # tie in row 2: lowest index (1) wins
    c.draft_tokens[0] = [2, 5, 6]
    r = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, 0.0, None)
    assert r["accept_len"][0] == 2
    assert list(r["tokens"][0]) == [2, 5, 1, -1]


# ------------------------------------------------------------------ bad input
def test_invalid_requests_are_marked():
    c = specsynth.make_verify_case("tiny", B=6)
    c.verify_len[1] = c.gamma + 1
    c.draft_tokens[2, 0] = c.V
    c.uniforms[3, c.gamma] = 1.0
    c.target[4, 2, 5] = np.nan
    c.draft[5, 1, :] = -np.inf
    r = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, c.T, c.uniforms)
    assert list(r["status"]) == [0, oracle.ERR_VERIFY_LEN, oracle.ERR_TOKEN, oracle.ERR_UNIFORM,
                                 oracle.ERR_NONFINITE, oracle.ERR_NONFINITE]
    assert r["accept_len"][0] >= 0
    assert (r["accept_len"][1:] == -1).all()
    assert (r["tokens"][1:] == -1).all()


def test_rows_beyond_verify_len_are_not_read():
    c = specsynth.make_verify_case("tiny", B=2)
    c.verify_len[:] = 1
    c.target[:, 2:] = np.nan
    c.draft[:, 1:] = np.nan
    c.draft_tokens[:, 1:] = -5
    r = oracle.verify(c.target, c.draft, c.dtype, c.draft_tokens, c.verify_len, c.T, c.uniforms)
    assert (r["status"] == 0).all()
    assert (r["accept_len"] <= 1).all()
