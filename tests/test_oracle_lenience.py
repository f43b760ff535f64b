"""Oracle pins for lenience [magicnet §8].

The page relaxes the acceptance test with a factor 0 < beta <= 1,
a = min(1, p / (beta q)); beta = 1 is the lossless rule, and no token is ever
drawn with more than 1/beta times its true probability.  The residual after a
rejection is the oracle's reading R12, (p - beta q)+ / Z_beta.

Pins (each checks the oracle against a statement of the page or a
consequence of the mathematics, not against a retyped formula):

* beta = 1 gives exactly the lossless results (same tokens, counts, a_i, Z).
* Exact single-position law, by enumeration of the draft token and of the
  uniform intervals: it sums to 1, P(x) <= p(x) / beta for every token (the
  page's guarantee), the bound is reached by every token with
  0 < p(x) <= beta q(x), and beta = 1 reproduces p.
* The acceptance rate grows as beta shrinks and equals sum min(p, q) at
  beta = 1 [rainlin §2]; once beta <= min p/q over the draft's support every
  draft is accepted and the output law is q.
* After a rejection the drawable tokens are exactly {x : p(x) > beta q(x)}.
* The page's table of beta values and their amplification bounds
  (tests/golden/magicnet_8_lenience.json).
"""
import numpy as np
import pytest

import oracle
from conftest import load_golden

T1 = (1.0, 0, 1.0)
BETAS = (1.0, 0.9, 0.6, 0.5, 0.3, 0.1)


def logits_of(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, dtype=np.float64))


def random_dist(rng, V, zero_frac=0.0):
    p = rng.dirichlet(np.ones(V))
    if zero_frac:
        mask = rng.random(V) < zero_frac
        if mask.all():
            mask[rng.integers(V)] = False
        p = np.where(mask, 0.0, p)
        p /= p.sum()
    return p


def first_token_law(p, q, beta):
    """Exact law of the first emitted token (gamma = 1) and the acceptance rate.

    Enumerates the draft token d ~ q, the accept / reject interval of u_accept
    and, on a rejection, every interval of u_sample that selects a token.
    """
    V = len(p)
    target = np.stack([logits_of(p), logits_of(p)])
    draft = logits_of(q)[None]
    law = np.zeros(V)
    accept = 0.0
    for d in range(V):
        if q[d] == 0.0:
            continue
        toks = np.array([d])
        probe = oracle.verify_sample_sequence(target, draft, toks, np.zeros(1), 0.5, T1, T1,
                                              1, 1, False, lenience=beta)
        a = float(probe.accept_prob[0])
        if a > 0.0:
            assert probe.num_accepted == 1 and probe.tokens[0] == d
            law[d] += q[d] * a
            accept += q[d] * a
        u_rej = np.array([(1.0 + a) / 2])
        if u_rej[0] < 1.0:        # else the reject interval is below one ulp (mass < 1e-16)
            res = oracle.verify_sample_sequence(target, draft, toks, u_rej, 0.5, T1, T1, 1, 1,
                                                False, keep_cdf=True, lenience=beta)
            assert res.num_accepted == 0
            cdf = res.sample_cdf
            lo = np.concatenate([[0.0], cdf[:-1]])
            for x in range(V):
                width = cdf[x] - lo[x]
                if width <= 0.0:
                    continue
                r = oracle.verify_sample_sequence(target, draft, toks, u_rej, (lo[x] + cdf[x]) / 2,
                                                  T1, T1, 1, 1, False, lenience=beta)
                assert r.tokens[0] == x
                law[x] += q[d] * (1.0 - a) * width
    return law, accept


def test_beta_one_is_lossless():
    rng = np.random.default_rng(81)
    B, G, V = 12, 4, 40
    target = rng.normal(0.0, 2.0, (B, G + 1, V))
    draft = target[:, :G] + rng.normal(0.0, 1.0, (B, G, V))
    tokens = rng.integers(0, V, (B, G))
    ua, us = rng.random((B, G)), rng.random(B)
    gam = rng.integers(0, G + 1, B)
    onehot = rng.random(B) < 0.3
    for params in ((1.0, 0, 1.0), (0.7, 8, 0.9)):
        base = oracle.verify_sample(target, draft, tokens, ua, us, params, params, gam, onehot)
        one = oracle.verify_sample(target, draft, tokens, ua, us, params, params, gam, onehot,
                                   lenience=1.0)
        np.testing.assert_array_equal(base.tokens, one.tokens)
        np.testing.assert_array_equal(base.num_accepted, one.num_accepted)
        np.testing.assert_array_equal(base.accept_prob, one.accept_prob)
        np.testing.assert_array_equal(base.residual_Z, one.residual_Z)
        np.testing.assert_array_equal(base.status, one.status)


@pytest.mark.parametrize("beta", BETAS)
def test_single_position_law_respects_the_bound(beta):
    rng = np.random.default_rng(int(beta * 1000) + 7)
    for trial in range(25):
        V = int(rng.integers(2, 7))
        p = random_dist(rng, V, 0.25 if trial % 3 == 1 else 0.0)
        q = random_dist(rng, V, 0.25 if trial % 3 == 2 else 0.0)
        law, _ = first_token_law(p, q, beta)
        assert abs(law.sum() - 1.0) < 1e-12
        assert np.all(law <= p / beta + 1e-12)                 # the page's guarantee
        tight = (p > 0.0) & (p <= beta * q - 1e-9)
        np.testing.assert_allclose(law[tight], p[tight] / beta, rtol=1e-11, atol=0)
        if beta == 1.0:
            np.testing.assert_allclose(law, p, atol=1e-12)      # lossless [wrblog §5.1]


def test_acceptance_grows_as_beta_shrinks():
    rng = np.random.default_rng(83)
    for _ in range(20):
        V = int(rng.integers(2, 7))
        p, q = random_dist(rng, V), random_dist(rng, V)
        rates = [first_token_law(p, q, beta)[1] for beta in BETAS]
        assert abs(rates[0] - np.minimum(p, q).sum()) < 1e-12  # alpha = sum min(p, q)
        assert all(r1 <= r2 + 1e-15 for r1, r2 in zip(rates, rates[1:]))
        beta_all = float(np.min(p[q > 0] / q[q > 0]))           # every draft accepted from here down
        if 0.0 < beta_all <= 1.0:
            for beta in (beta_all, beta_all / 2):
                law, rate = first_token_law(p, q, beta)
                assert abs(rate - 1.0) < 1e-12
                np.testing.assert_allclose(law, q, atol=1e-12)


@pytest.mark.parametrize("beta", (0.9, 0.5, 0.3))
def test_residual_support(beta):
    rng = np.random.default_rng(int(beta * 100) + 91)
    checked = 0
    for _ in range(30):
        V = int(rng.integers(3, 9))
        p, q = random_dist(rng, V), random_dist(rng, V)
        if np.any(np.abs(p - beta * q) < 1e-9):
            continue
        target = np.stack([logits_of(p), logits_of(p)])
        draft = logits_of(q)[None]
        for d in range(V):
            probe = oracle.verify_sample_sequence(target, draft, np.array([d]), np.zeros(1), 0.5,
                                                  T1, T1, 1, 1, False, lenience=beta)
            a = float(probe.accept_prob[0])
            if a >= 1.0:
                continue
            res = oracle.verify_sample_sequence(target, draft, np.array([d]), np.array([(1 + a) / 2]),
                                                0.5, T1, T1, 1, 1, False, keep_cdf=True, lenience=beta)
            cdf = res.sample_cdf
            width = np.diff(np.concatenate([[0.0], cdf]))
            np.testing.assert_array_equal(width > 0, p > beta * q)
            checked += 1
    assert checked > 20


def test_one_hot_draft_with_lenience():
    """q is a delta at d: a = min(1, p(d) / beta), and a rejection never redraws d."""
    rng = np.random.default_rng(97)
    V = 6
    p = random_dist(rng, V)
    target = np.stack([logits_of(p), logits_of(p)])
    for beta in BETAS:
        for d in range(V):
            r = oracle.verify_sample_sequence(target, None, np.array([d]), np.zeros(1), 0.5, T1, T1,
                                              1, 1, True, keep_cdf=True, lenience=beta)
            assert abs(r.accept_prob[0] - min(1.0, p[d] / beta)) < 1e-12
            rej = oracle.verify_sample_sequence(target, None, np.array([d]), np.array([0.999999]), 0.5,
                                                T1, T1, 1, 1, True, keep_cdf=True, lenience=beta)
            if rej.num_accepted == 0:
                assert rej.tokens[0] != d


def test_page_table():
    g = load_golden("magicnet_8_lenience.json")
    rng = np.random.default_rng(101)
    for row in g["table"]:
        beta = row["beta"]
        assert abs(1.0 / beta - row["max_amplification_printed"]) < 0.5   # the printed bound, rounded
        worst = 0.0
        for _ in range(20):
            V = int(rng.integers(2, 6))
            p, q = random_dist(rng, V), random_dist(rng, V)
            law, _ = first_token_law(p, q, beta)
            worst = max(worst, float(np.max(law[p > 0] / p[p > 0])))
        assert worst <= 1.0 / beta + 1e-9
        if beta < 1.0:
            assert worst > 1.0                                   # the relaxation does amplify


def test_lenience_range():
    target = np.zeros((2, 4))
    for bad in (0.0, -0.5, 1.5, np.nan):
        with pytest.raises(ValueError):
            oracle.verify_sample_sequence(target, None, np.array([0]), np.zeros(1), 0.5, T1, T1,
                                          1, 1, True, lenience=bad)
