"""Oracle pins: the worked examples the pages print (fixtures under tests/golden/)."""
import numpy as np

import oracle
from conftest import load_golden

T1 = (1.0, 0, 1.0)   # temperature 1, no top-k, no top-p: p is softmax(log p) = p


def logits_of(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, dtype=np.float64))


def run_one(p, q, draft, u_acc, u_samp):
    """One draft position through the full oracle (gamma = 1)."""
    target = np.stack([logits_of(p), logits_of(p)])   # row 2 is the bonus row
    dr = logits_of(q)[None, :]
    return oracle.verify_sample_sequence(target, dr, np.array([draft]), np.array([u_acc]), u_samp,
                                         T1, T1, 1, 1, False, keep_cdf=True)


def test_wrblog_three_token_example():
    g = load_golden("wrblog_4_3_three_token_example.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    for i, name in enumerate(g["tokens"]):
        a, zq = oracle.acceptance_probability(p[i], q[i])
        assert not zq
        assert abs(a - g["accept_probability"][name]) < 1e-12
        # through the full pipeline: accept_prob output for draft token i
        r = run_one(p, q, i, 0.0, 0.5)
        assert abs(r.accept_prob[0] - g["accept_probability"][name]) < 1e-12
    assert abs(oracle.acceptance_rate(p, q) - g["acceptance_rate"]) < 1e-12
    np.testing.assert_allclose(p - q, g["p_minus_q"], atol=1e-12)
    w = oracle.residual_weights(p, q)
    np.testing.assert_allclose(w / w.sum(), g["residual"], atol=1e-12)
    # B (index 1) rejected -> the replacement is always A, whatever u_sample is
    for u_samp in (0.0, 0.3, 0.999999):
        r = run_one(p, q, 1, 0.61, u_samp)
        assert r.num_accepted == 0 and r.tokens[0] == 0
        assert abs(r.residual_Z - 0.25) < 1e-12
    # B accepted when u < 0.6
    r = run_one(p, q, 1, 0.59, 0.5)
    assert r.num_accepted == 1 and r.tokens[0] == 1


def test_baisen_mat_sat_ran():
    g = load_golden("baisen_4_mat_sat_ran.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    d = g["tokens"].index(g["draft"])
    r = run_one(p, q, d, 0.0, 0.5)
    assert abs(r.accept_prob[0] - g["accept_probability_exact"]) < 1e-12
    assert round(r.accept_prob[0], 2) == g["accept_probability_printed"]
    w = oracle.residual_weights(p, q)
    np.testing.assert_allclose(w / w.sum(), g["residual"], atol=1e-12)
    r = run_one(p, q, d, 0.9, 0.77)   # rejected: always "sat"
    assert r.num_accepted == 0 and g["tokens"][r.tokens[0]] == "sat"


def test_baisen_counterexample_accepts_non_argmax():
    g = load_golden("baisen_6_counterexample.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    d = g["tokens"].index(g["draft"])
    r = run_one(p, q, d, 0.0, 0.5)
    assert abs(r.accept_prob[0] - g["accept_probability"]) < 1e-12
    assert g["tokens"][int(np.argmax(p))] == g["target_argmax"]
    assert r.num_accepted == 1 and g["tokens"][r.tokens[0]] == g["draft"]


def test_wrblog_greedy_example():
    g = load_golden("wrblog_7_1_greedy.json")
    z = logits_of(g["p"])
    d = g["tokens"].index(g["draft"])
    r = oracle.verify_greedy_sequence(np.stack([z, z]), np.array([d]), 1, 1)
    assert r.num_accepted == g["num_accepted"]
    assert g["tokens"][r.tokens[0]] == g["emitted"]
    assert r.tokens[1] == -1


def test_baisen_greedy_chain():
    g = load_golden("baisen_2_greedy_chain.json")
    vocab = g["vocab"]
    V = len(vocab)
    gamma = len(g["drafts"])
    target = np.full((gamma + 1, V), -1.0)
    for i, top in enumerate(g["target_top1"]):
        target[i, vocab.index(top)] = 3.0
    target[gamma, vocab.index("sat")] = 3.0          # unspecified on the page; never reached
    drafts = np.array([vocab.index(t) for t in g["drafts"]])
    r = oracle.verify_greedy_sequence(target, drafts, gamma, gamma)
    assert r.num_accepted == g["num_accepted"]
    assert [vocab[t] for t in r.tokens[: r.num_accepted + 1]] == g["committed"]


def test_strict_less_than_rule():
    """Accept iff u < a (the demo's comparison): u == a rejects."""
    target = np.array([[0.0, 0.0], [0.0, 0.0]])      # p = [1/2, 1/2] exactly
    draft = np.array([[0.0, -np.inf]])               # q = [1, 0]  -> a(0) = 1/2 exactly
    kw = dict(target_params=T1, draft_params=T1, gamma_b=1, gamma_max=1, one_hot=False)
    r = oracle.verify_sample_sequence(target, draft, np.array([0]), np.array([0.5]), 0.1, **kw)
    assert r.accept_prob[0] == 0.5 and r.num_accepted == 0
    r = oracle.verify_sample_sequence(target, draft, np.array([0]), np.array([np.nextafter(0.5, 0)]), 0.1, **kw)
    assert r.num_accepted == 1


def test_inverse_cdf_vocabulary_order():
    w = np.array([0.2, 0.0, 0.3, 0.5])
    # C = [0.2, 0.2, 0.5, 1.0]; first C > u
    assert oracle.inverse_cdf(w, 0.0)[0] == 0
    assert oracle.inverse_cdf(w, 0.19)[0] == 0
    assert oracle.inverse_cdf(w, 0.2)[0] == 2       # boundary goes up; zero-weight token 1 skipped
    assert oracle.inverse_cdf(w, 0.49)[0] == 2
    assert oracle.inverse_cdf(w, 0.5)[0] == 3
    tok, lo, hi = oracle.inverse_cdf(w, 0.7)
    assert tok == 3 and abs(lo - 0.5) < 1e-15 and hi == 1.0


def test_zero_q_rule_and_one_hot():
    # q(d) = 0 is reachable only for a draft not sampled from q; flag it (a = 1 if p(d) > 0)
    target = np.log(np.array([[0.5, 0.5], [0.5, 0.5]]))
    draft = np.array([[0.0, -np.inf]])
    r = oracle.verify_sample_sequence(target, draft, np.array([1]), np.array([0.999]), 0.1,
                                      T1, T1, 1, 1, False)
    assert r.accept_prob[0] == 1.0 and r.num_accepted == 1
    assert r.status & oracle.SEQ_FLAG_ZERO_Q
    # one-hot draft: q = delta, acceptance = p(d)  [baisen §6 greedy-as-special-case algebra]
    r = oracle.verify_sample_sequence(target, None, np.array([1]), np.array([0.49]), 0.1,
                                      T1, T1, 1, 1, True)
    assert abs(r.accept_prob[0] - 0.5) < 1e-12 and r.num_accepted == 1
    r = oracle.verify_sample_sequence(target, None, np.array([1]), np.array([0.51]), 0.1,
                                      T1, T1, 1, 1, True)
    # rejected: residual (p - delta_1)+ puts all mass on token 0
    assert r.num_accepted == 0 and r.tokens[0] == 0 and abs(r.residual_Z - 0.5) < 1e-12


def test_error_statuses_commit_nothing():
    V, G = 4, 2
    tgt = np.zeros((G + 1, V))
    dft = np.zeros((G, V))
    toks = np.array([1, 2])
    ua = np.array([0.5, 0.5])
    kw = dict(target_params=T1, draft_params=T1, gamma_max=G, one_hot=False)
    assert oracle.verify_sample_sequence(tgt, dft, toks, ua, 0.5, gamma_b=3, **kw).status == oracle.SEQ_BAD_LENGTH
    assert oracle.verify_sample_sequence(tgt, dft, np.array([1, 4]), ua, 0.5, gamma_b=2, **kw).status == oracle.SEQ_BAD_TOKEN
    assert oracle.verify_sample_sequence(tgt, dft, toks, ua, 1.0, gamma_b=2, **kw).status == oracle.SEQ_BAD_UNIFORM
    bad = tgt.copy(); bad[2, 1] = np.nan
    r = oracle.verify_sample_sequence(bad, dft, toks, ua, 0.5, gamma_b=2, **kw)
    assert r.status == oracle.SEQ_NONFINITE and r.num_accepted == -1 and (r.tokens == -1).all()
    bad = tgt.copy(); bad[1, 0] = np.inf
    assert oracle.verify_sample_sequence(bad, dft, toks, ua, 0.5, gamma_b=2, **kw).status == oracle.SEQ_NONFINITE
    bad = dft.copy(); bad[0] = -np.inf
    assert oracle.verify_sample_sequence(tgt, bad, toks, ua, 0.5, gamma_b=2, **kw).status == oracle.SEQ_EMPTY_SUPPORT
    # rows beyond gamma_b are never read
    bad = tgt.copy(); bad[2] = np.nan
    assert oracle.verify_sample_sequence(bad, dft, toks, ua, 0.5, gamma_b=1, **kw).status == oracle.SEQ_OK
    # gamma_b = 0: just the bonus draw from p_1
    r = oracle.verify_sample_sequence(tgt, dft, toks, ua, 0.6, gamma_b=0, **kw)
    assert r.num_accepted == 0 and r.tokens[0] == 2 and r.tokens[1] == -1


def test_runtime_invariants_no_draft_after_rejection():
    """[wrblog §13.2, §14.3]: drafts after the first rejection never reach the output;
    the emitted block is the accepted prefix plus exactly one target token."""
    rng = np.random.default_rng(5)
    V, G = 6, 4
    for _ in range(200):
        tgt = rng.normal(0, 1.5, size=(G + 1, V))
        dft = tgt[:G] + rng.normal(0, 1.0, size=(G, V))
        toks = rng.integers(0, V, size=G)
        ua = rng.random(G)
        gb = int(rng.integers(0, G + 1))
        r = oracle.verify_sample_sequence(tgt, dft, toks, ua, float(rng.random()), (0.9, 0, 1.0),
                                          (1.1, 3, 0.95), gb, G, False)
        n = r.num_accepted
        assert 0 <= n <= gb
        assert (r.tokens[:n] == toks[:n]).all()
        assert 0 <= r.tokens[n] < V
        assert (r.tokens[n + 1:] == -1).all()
        # the scan stopped exactly at the first u_i >= a_i
        assert all(ua[i] < r.accept_prob[i] for i in range(n))
        assert n == gb or ua[n] >= r.accept_prob[n]
