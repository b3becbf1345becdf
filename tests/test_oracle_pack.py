"""Pins of the oracle's dense packing of ragged prefixes (AngelSpec §4.2,
"Packing and correctness")."""
import numpy as np

import oracle


def test_pack_rows_by_hand():
    """verify lengths [2, 0, 3, 1] (gamma 3): target rows 3, 1, 4, 2 and draft
    rows 2, 0, 3, 1, one request after another."""
    r = oracle.pack_rows([2, 0, 3, 1], 3)
    assert r["rc"] == 0
    assert list(r["target_row"]) == [0, 3, 4, 8]
    assert list(r["draft_row"]) == [0, 2, 2, 5]
    assert (r["K_target"], r["K_draft"]) == (10, 6)


def test_invalid_lengths_take_no_rows():
    r = oracle.pack_rows([1, -1, 5, 2], 4)
    assert list(r["target_row"]) == [0, 2, 2, 2]
    assert list(r["draft_row"]) == [0, 1, 1, 1]
    assert (r["K_target"], r["K_draft"]) == (5, 3)


def test_packing_is_a_bijection_onto_the_kept_rows():
    """Every kept (request, position) gets its own packed row, and the packed
    rows are exactly 0..K-1: target K = B + sum ell = the budget N."""
    rng = np.random.default_rng(3)
    for _ in range(50):
        B, gamma = int(rng.integers(1, 300)), int(rng.integers(0, 33))
        vl = rng.integers(0, gamma + 1, B).astype(np.int32)
        r = oracle.pack_rows(vl, gamma)
        assert r["K_target"] == int((vl + 1).sum()) and r["K_draft"] == int(vl.sum())
        t = np.concatenate([r["target_row"][b] + np.arange(vl[b] + 1) for b in range(B)])
        d = np.concatenate([r["draft_row"][b] + np.arange(vl[b]) for b in range(B)] + [np.zeros(0, int)])
        assert sorted(t) == list(range(r["K_target"]))
        assert sorted(d) == list(range(r["K_draft"]))
