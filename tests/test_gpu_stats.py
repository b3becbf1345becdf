"""Statistical checks of the CUDA path itself: over 10^6 replicated requests
the emitted tokens follow the target distribution (chi-square), acceptance per
position matches the overlap, and the mean accepted length matches the closed
form."""
import numpy as np
import pytest
from scipy import stats

import specsynth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def run():
    import torch
    import speculative_decoding_verification_softmax_gb300 as sv
    sv.build()
    rng = np.random.default_rng(2025)
    gamma, V, B = 3, 5, 1_000_000
    P = rng.dirichlet(np.ones(V), size=gamma + 1)
    Q = rng.dirichlet(np.ones(V), size=gamma)
    case = specsynth.make_replicated_case(P, Q, B, seed_tokens=81, seed_uniforms=82, dtype="f32")
    t, d, x, vl, u = H.to_device(case)
    toks, lens = [], []
    step = sv.MAX_BATCH
    ws = sv.alloc_verify_workspace(step, gamma, V, sv.F32)
    for b0 in range(0, B, step):
        b1 = min(B, b0 + step)
        tok, n, _ = sv.verify(t[b0:b1], d[b0:b1], x[b0:b1], vl[b0:b1], 1.0, u[b0:b1], workspace=ws)
        toks.append(tok)
        lens.append(n)
    assert sv.read_status(ws) == 0
    tok = torch.cat(toks).cpu().numpy()
    n = torch.cat(lens).cpu().numpy()
    return P, Q, tok, n


def _chi2_p(counts, probs):
    return stats.chisquare(counts, probs * counts.sum()).pvalue


def test_first_token_distribution(run):
    P, Q, tok, n = run
    assert _chi2_p(np.bincount(tok[:, 0], minlength=5), P[0]) > 1e-4


def test_second_token_given_first_accepted(run):
    P, Q, tok, n = run
    sel = n >= 1
    assert _chi2_p(np.bincount(tok[sel, 1], minlength=5), P[1]) > 1e-4


def test_bonus_token_distribution(run):
    P, Q, tok, n = run
    sel = n == 3
    assert _chi2_p(np.bincount(tok[sel, 3], minlength=5), P[3]) > 1e-4


def test_acceptance_and_expected_length(run):
    P, Q, tok, n = run
    alpha = np.minimum(P[:3], Q).sum(axis=1)
    for j in range(3):
        reached = n >= j
        acc = (n[reached] > j).mean()
        assert abs(acc - alpha[j]) < 4 * np.sqrt(alpha[j] * (1 - alpha[j]) / reached.sum())
    expect = sum(np.prod(alpha[: j + 1]) for j in range(3))
    assert abs(n.mean() - expect) < 4 * n.std() / np.sqrt(n.size)
