"""Oracle pins that follow from the mathematics on the pages.

* Identities: Z = sum (p-q)+ = sum (q-p)+ = 1 - sum min(p,q) = P(reject),
  min(p,q) + (p-q)+ = p, acceptance = 1 - TV(p,q).
  [rainlin §2; baisen §5; magicnet §3; wrblog §4.2, §5.1]
* Exact output law by exhaustive enumeration of drafts and of the uniform
  intervals: one position reproduces p; several rounds reproduce the target's
  autoregressive law.  [wrblog §5.1, §6.1; rainlin §2]
* Tokens per round under i.i.d. acceptance: P(T=k) = a^{k-1}(1-a) for k <= g,
  P(T=g+1) = a^g, E[T] = (1 - a^{g+1}) / (1 - a), and the printed values.
  [magicnet §4, §9; rainlin §3; wrblog §10]
* The single-position demo's statistics.  [wrblog §8]
"""
import functools

import numpy as np
import pytest

import oracle
from conftest import load_golden

T1 = (1.0, 0, 1.0)


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


def test_residual_identities():
    rng = np.random.default_rng(10)
    for trial in range(200):
        V = int(rng.integers(2, 50))
        p = random_dist(rng, V, 0.3 if trial % 2 else 0.0)
        q = random_dist(rng, V, 0.3 if trial % 3 else 0.0)
        z_pos = oracle.residual_weights(p, q).sum()
        z_neg = oracle.residual_weights(q, p).sum()
        alpha = oracle.acceptance_rate(p, q)
        tv = 0.5 * np.abs(p - q).sum()
        assert abs(z_pos - z_neg) < 1e-12
        assert abs(z_pos - (1.0 - alpha)) < 1e-12
        assert abs(alpha - (1.0 - tv)) < 1e-12
        # P(reject) by the law of total probability over the proposed token
        p_reject = sum(q[x] * (1.0 - oracle.acceptance_probability(p[x], q[x])[0])
                       for x in range(V) if q[x] > 0)
        assert abs(p_reject - z_pos) < 1e-12
        np.testing.assert_allclose(np.minimum(p, q) + oracle.residual_weights(p, q), p, atol=1e-15)


def one_round_law(p_of, q_of, prefix, V, gamma):
    """Law of the block emitted by one verification round from context ``prefix``.

    p_of(ctx), q_of(ctx) give the target / draft probability vectors for a context tuple.
    Returns {emitted_tuple: probability}.
    """
    law = {}
    for drafts in np.ndindex(*([V] * gamma)):
        w_d = 1.0
        ctx = prefix
        for t in drafts:
            w_d *= q_of(ctx)[t]
            ctx = ctx + (t,)
        if w_d == 0.0:
            continue
        target = np.stack([logits_of(p_of(prefix + drafts[:i])) for i in range(gamma + 1)])
        draft = np.stack([logits_of(q_of(prefix + drafts[:i])) for i in range(gamma)])
        toks = np.array(drafts)
        probe = oracle.verify_sample_sequence(target, draft, toks, np.zeros(gamma), 0.5,
                                              T1, T1, gamma, gamma, False)
        a = probe.accept_prob[:gamma]
        for j in range(gamma + 1):                 # j = first rejected position; gamma = none
            if j < gamma:
                w_acc = np.prod(a[:j]) * (1.0 - a[j])
                u_acc = np.array([a[i] / 2 for i in range(j)] + [(1.0 + a[j]) / 2] +
                                 [0.5] * (gamma - j - 1))
            else:
                w_acc = np.prod(a)
                u_acc = a / 2
            if w_acc == 0.0:
                continue
            res = oracle.verify_sample_sequence(target, draft, toks, u_acc, 0.5, T1, T1,
                                                gamma, gamma, False, keep_cdf=True)
            assert res.num_accepted == j
            cdf = res.sample_cdf
            lo = np.concatenate([[0.0], cdf[:-1]])
            for x in range(V):
                width = cdf[x] - lo[x]
                if width <= 0:
                    continue
                r = oracle.verify_sample_sequence(target, draft, toks, u_acc, (lo[x] + cdf[x]) / 2,
                                                  T1, T1, gamma, gamma, False)
                assert r.tokens[j] == x
                block = tuple(int(t) for t in r.tokens[: j + 1])
                law[block] = law.get(block, 0.0) + w_d * w_acc * width
    return law


def sequence_law(p_of, q_of, V, gamma, L):
    """Law of the first L emitted tokens when rounds repeat from the growing prefix."""
    @functools.lru_cache(maxsize=None)
    def law_from(prefix):
        out = {}
        if len(prefix) >= L:
            return {prefix[:L]: 1.0}
        for block, w in one_round_law(p_of, q_of, prefix, V, gamma).items():
            for seq, w2 in law_from(prefix + block).items():
                out[seq] = out.get(seq, 0.0) + w * w2
        return out
    return law_from(())


@pytest.mark.parametrize("V,gamma,zeros,seed", [(3, 1, 0.0, 0), (3, 2, 0.0, 1), (4, 2, 0.3, 2),
                                                (3, 3, 0.25, 3)])
def test_multi_token_law_equals_target_autoregressive_law(V, gamma, zeros, seed):
    rng = np.random.default_rng(100 + seed)
    tables_p, tables_q = {}, {}

    def p_of(ctx):
        if ctx not in tables_p:
            tables_p[ctx] = random_dist(rng, V, zeros)
        return tables_p[ctx]

    def q_of(ctx):
        if ctx not in tables_q:
            tables_q[ctx] = random_dist(rng, V, zeros)
        return tables_q[ctx]

    L = gamma + 1
    law = sequence_law(p_of, q_of, V, gamma, L)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    for seq in np.ndindex(*([V] * L)):
        expect = 1.0
        for t in range(L):
            expect *= p_of(tuple(seq[:t]))[seq[t]]
        assert abs(law.get(tuple(seq), 0.0) - expect) < 1e-12, (seq, law.get(tuple(seq)), expect)


def single_position_law(p, q):
    V = len(p)
    law = one_round_law(lambda c: p, lambda c: q, (), V, 1)
    out = np.zeros(V)
    for block, w in law.items():
        out[block[0]] += w
    return out


def test_single_position_output_law_is_p():
    g = load_golden("wrblog_4_3_three_token_example.json")
    np.testing.assert_allclose(single_position_law(np.array(g["p"]), np.array(g["q"])), g["p"],
                               atol=1e-12)
    rng = np.random.default_rng(11)
    for _ in range(10):
        V = int(rng.integers(2, 7))
        p, q = random_dist(rng, V, 0.2), random_dist(rng, V, 0.2)
        np.testing.assert_allclose(single_position_law(p, q), p, atol=1e-12)


def tokens_per_round_law(p, q, gamma):
    """Exact law of T (tokens emitted in one round) for position-independent p, q."""
    law = one_round_law(lambda c: p, lambda c: q, (), len(p), gamma)
    out = np.zeros(gamma + 2)
    for block, w in law.items():
        out[len(block)] += w
    return out


def dists_with_alpha(alpha):
    """p, q over 3 tokens with sum min(p, q) = alpha exactly in exact arithmetic."""
    p = np.array([alpha, 1.0 - alpha, 0.0])
    q = np.array([1.0, 0.0, 0.0])
    return p, q


def closed_form_E(alpha, gamma):
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


@pytest.mark.parametrize("gamma", [1, 2, 4, 5])
@pytest.mark.parametrize("alpha", [0.4, 0.6, 0.8, 0.9])
def test_truncated_geometric_tokens_per_round(alpha, gamma):
    rng = np.random.default_rng(int(alpha * 100) + gamma)
    for p, q in [dists_with_alpha(alpha)]:
        law = tokens_per_round_law(p, q, gamma)
        for k in range(1, gamma + 1):
            assert abs(law[k] - alpha ** (k - 1) * (1 - alpha)) < 1e-12
        assert abs(law[gamma + 1] - alpha ** gamma) < 1e-12
        E = (np.arange(gamma + 2) * law).sum()
        assert abs(E - closed_form_E(alpha, gamma)) < 1e-12
    # a generic pair with the same overlap gives the same law (only alpha matters)
    V = 4
    p = random_dist(rng, V)
    q = random_dist(rng, V)
    a = oracle.acceptance_rate(p, q)
    law = tokens_per_round_law(p, q, min(gamma, 2))
    E = (np.arange(law.size) * law).sum()
    assert abs(E - closed_form_E(a, min(gamma, 2))) < 1e-12


def test_printed_expected_token_values():
    g = load_golden("magicnet_4_expected_tokens.json")

    def enumerated_E(alpha, gamma):
        p, q = dists_with_alpha(alpha)
        law = tokens_per_round_law(p, q, gamma)
        return (np.arange(gamma + 2) * law).sum()

    for gamma_s, row in g["table"].items():
        gamma = int(gamma_s)
        for alpha, printed in zip(g["alphas"], row):
            val = enumerated_E(alpha, gamma)
            assert round(val, g["table_decimals"]) == pytest.approx(printed, abs=1e-9), (gamma, alpha)
    for w in g["worked"]:
        assert round(enumerated_E(w["alpha"], w["gamma"]), w["decimals"]) == pytest.approx(w["value"])
    for w in g["ideal_speedup_c0"]:
        val = enumerated_E(w["alpha"], w["gamma"])
        assert round(val, 2) == pytest.approx(w["value"])


def test_single_position_demo_statistics():
    """The demo draws d ~ q, accepts with min(1, p/q), else resamples the residual;
    the empirical output is ~p and the acceptance ~0.75 (binomial 5 sigma)."""
    g = load_golden("wrblog_8_demo.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    rng = np.random.default_rng(g["seed"])
    n = 40_000
    target = np.stack([logits_of(p), logits_of(p)])
    draft = logits_of(q)[None, :]
    counts = np.zeros(3)
    accepted = 0
    drafts = rng.choice(3, size=n, p=q)
    u = rng.random((n, 2))
    for t in range(n):
        r = oracle.verify_sample_sequence(target, draft, drafts[t:t + 1], u[t, :1], u[t, 1],
                                          T1, T1, 1, 1, False)
        counts[r.tokens[0]] += 1
        accepted += r.num_accepted
    freq = counts / n
    sig = np.sqrt(np.array(g["expected_output_distribution"]) * (1 - np.array(g["expected_output_distribution"])) / n)
    assert (np.abs(freq - g["expected_output_distribution"]) < 5 * sig).all(), freq
    a = g["expected_acceptance"]
    assert abs(accepted / n - a) < 5 * np.sqrt(a * (1 - a) / n)
