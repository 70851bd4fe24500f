"""Pins of the oracle's top-k / top-p sampling settings (CPU).

Every check stands on something other than the oracle's own formula: a hand-worked example, the
tie order, brute-force minimality of the top-p set, the greedy verifier (top-k = 1 turns
speculative sampling into greedy verification), and distribution preservation.
"""
import itertools
import json
import os

import numpy as np
import pytest
from scipy import stats

import oracle.specdec_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "top_p_example.json")))
    z = np.log(np.array(g["probabilities_by_token"]))
    for c in g["cases"]:
        keep = O.sampling_keep(z, 1.0, c["top_k"], c["top_p"])
        assert sorted(np.nonzero(keep)[0].tolist()) == c["kept"], c
        for tok, pv in c.get("p", {}).items():
            assert O.filtered_softmax(z, 1.0, c["top_k"], c["top_p"])[int(tok)] == pytest.approx(pv)


def test_ties_keep_lower_indices():
    z = np.array([1.0, 2.0, 1.0, 2.0, 1.0])
    assert np.nonzero(O.sampling_keep(z, 1.0, top_k=3))[0].tolist() == [0, 1, 3]
    # equal probabilities 1/3 each among three tied tokens: mass before the third is 2/3
    z = np.zeros(3)
    assert np.nonzero(O.sampling_keep(z, 1.0, top_p=0.6))[0].tolist() == [0, 1]
    assert np.nonzero(O.sampling_keep(z, 1.0, top_p=0.7))[0].tolist() == [0, 1, 2]


def test_top_p_set_is_minimal_by_brute_force():
    """The top-p set reaches top_p of the (top-k) mass, and no smaller set of tokens does."""
    rng = np.random.default_rng(5)
    for _ in range(60):
        V = int(rng.integers(2, 8))
        z = rng.normal(size=V) * 2
        T = float(rng.uniform(0.3, 2.0))
        k = int(rng.integers(0, V + 1))
        tp = float(rng.uniform(0.05, 0.99))
        keep = O.sampling_keep(z, T, k, tp)
        p = np.exp(z / T - (z / T).max())
        base = np.argsort(-z, kind="stable")[: (V if k <= 0 or k >= V else k)]
        mass = p[base].sum()
        assert p[keep].sum() >= tp * mass * (1 - 1e-12)
        n = int(keep.sum())
        for m in range(1, n):                      # no set of m < n tokens reaches top_p
            assert max(p[list(s)].sum() for s in itertools.combinations(base, m)) < tp * mass
        assert set(np.nonzero(keep)[0]) <= set(base.tolist())


def test_settings_off_give_plain_softmax():
    rng = np.random.default_rng(6)
    z = rng.normal(size=50)
    assert np.array_equal(O.filtered_softmax(z, 0.7), O.softmax(z, 0.7))
    assert np.array_equal(O.filtered_softmax(z, 0.7, top_k=50, top_p=1.0), O.softmax(z, 0.7))
    with pytest.raises(O.OracleError):
        O.sampling_keep(z, 0.7, top_p=0.0)


def test_top_k_one_is_greedy_verification():
    """With top-k = 1 both p and q are one-hot at their argmax: drafts that are the draft model's
    argmax are accepted exactly while they equal the target's argmax, and the replacement or bonus
    is the target's argmax -- the greedy verifier's result."""
    rng = np.random.default_rng(7)
    B, D, V = 40, 5, 30
    tl = rng.normal(size=(B, D + 1, V))
    dl = tl[:, :D] + rng.normal(scale=0.7, size=(B, D, V))
    draft = dl.argmax(-1).astype(np.int32)
    u = rng.random((B, D + 1))
    a, y, _, _ = O.verify_sample(tl, dl, draft, u, 0.8, top_k=1)
    ga, gy = O.verify_greedy(tl, draft)
    np.testing.assert_array_equal(a, ga)
    np.testing.assert_array_equal(y, gy)
    assert 0 < (a < D).mean() < 1


def test_filtered_sampling_preserves_the_filtered_target():
    """Drafts drawn from the filtered q: the first emitted token is distributed as the filtered p,
    and the acceptance probability is the overlap sum of min(p', q')."""
    rng = np.random.default_rng(8)
    V, n, T = 8, 40000, 0.9
    for k, tp in ((5, 1.0), (0, 0.8), (6, 0.7)):
        zp, zq = rng.normal(size=V), rng.normal(size=V)
        pf = O.filtered_softmax(zp, T, k, tp)
        qf = O.filtered_softmax(zq, T, k, tp)
        tl = np.broadcast_to(np.stack([zp, zp]), (n, 2, V))
        dl = np.broadcast_to(zq[None, None], (n, 1, V))
        draft = rng.choice(V, size=(n, 1), p=qf).astype(np.int32)
        u = rng.random((n, 2))
        a, y, _, _ = O.verify_sample(tl, dl, draft, u, T, top_k=k, top_p=tp)
        first = np.where(a >= 1, draft[:, 0], y)
        exp = pf * n
        mask = exp > 0
        assert (np.bincount(first, minlength=V)[~mask] == 0).all()
        assert stats.chisquare(np.bincount(first, minlength=V)[mask], exp[mask]).pvalue > 1e-3
        pacc = np.minimum(pf, qf).sum()
        assert abs((a == 1).mean() - pacc) < 4 * np.sqrt(pacc * (1 - pacc) / n)


def test_drafts_outside_the_kept_sets():
    """min(1, p/q) at the edges of the kept sets: a draft the target cannot emit (p(d) = 0) is
    rejected for every u, also when the draft model cannot emit it either (0/0); a draft outside
    the draft model's set only (q(d) = 0 < p(d)) is accepted for every u; the replacement after a
    rejection is always a token the target can emit."""
    zp = np.log(np.array([0.4, 0.3, 0.1, 0.1, 0.05, 0.05]))   # top-2 keeps {0, 1}
    zq = np.log(np.array([0.05, 0.4, 0.3, 0.1, 0.1, 0.05]))   # top-2 keeps {1, 2}
    tl = np.stack([zp, zp])[None]
    dl = zq[None, None]
    for d, want in ((4, 0), (5, 0), (2, 0), (0, 1)):
        for u0 in (0.0, 0.3, 0.999999):
            for u1 in (0.0, 0.5, 0.999999):
                a, y, _, _ = O.verify_sample(tl, dl, np.array([[d]]), np.array([[u0, u1]]), 1.0,
                                             top_k=2)
                assert a[0] == want, (d, u0)
                assert y[0] in (0, 1)
    # the same 0/0 case without sampling settings: both scores -inf
    zp2, zq2 = zp.copy(), zq.copy()
    zp2[4] = zq2[4] = -np.inf
    a, y, _, _ = O.verify_sample(np.stack([zp2, zp2])[None], zq2[None, None], np.array([[4]]),
                                 np.array([[0.0, 0.5]]), 1.0)
    assert a[0] == 0 and y[0] != 4


def test_planted_mistakes_are_caught(monkeypatch):
    """Mistakes planted in the oracle fail the pins above: ties ordered by higher index, and the
    top-p cut taken on the mass including the token instead of the mass before it."""
    g = json.load(open(os.path.join(GOLDEN, "top_p_example.json")))
    z6 = np.log(np.array(g["probabilities_by_token"]))
    zt = np.array([1.0, 2.0, 1.0, 2.0, 1.0])
    with monkeypatch.context() as m:
        m.setattr(O, "_sort_order", lambda z: np.lexsort((-np.arange(len(z)), -z)))
        assert np.nonzero(O.sampling_keep(zt, 1.0, top_k=3))[0].tolist() != [0, 1, 3]
    with monkeypatch.context() as m:
        real_cumsum = np.cumsum

        def inclusive(x, *a, **k):                 # "before" becomes "including the token"
            c = real_cumsum(x, *a, **k)
            return np.concatenate((c[1:], c[-1:]))
        m.setattr(O.np, "cumsum", inclusive)
        kept = sorted(np.nonzero(O.sampling_keep(z6, 1.0, 0, 0.6))[0].tolist())
        assert kept != [0, 3]
    assert sorted(np.nonzero(O.sampling_keep(z6, 1.0, 0, 0.6))[0].tolist()) == [0, 3]


def test_margin_helper():
    z = np.log(np.array([0.5, 0.3, 0.2]))
    assert O.top_p_margin(z, 1.0, 0, 0.75) == pytest.approx(0.05)   # preceding masses 0, .5, .8
    assert O.top_p_margin(z, 1.0, 0, 1.0) == np.inf
