"""Pins for the early-exit greedy oracle (reading R11).

The sequential verifier of [wrblog §6] reads position after position and
stops at the first draft the target rejects; with the greedy test of
[wrblog §7.1] that is the first d_i != argmax z_i.  These tests pin the
early-exit oracle to the page examples, to the all-rows greedy oracle on
valid inputs, to its error semantics (rows after the stop are never read),
and to the truncated-geometric law of the rows it reads [magicnet §4].
"""
import itertools

import numpy as np
import pytest

import oracle
from conftest import load_golden


def logits_of(p):
    return np.log(np.asarray(p, dtype=np.float64))


def test_baisen_chain_never_reads_the_unspecified_row():
    """[baisen §2]: the page gives no top-1 for the fifth (bonus) position.  The
    sequential verifier stops at the fourth position, so that row may hold
    anything -- even NaN -- while the all-rows verifier has to fail on it."""
    g = load_golden("baisen_2_greedy_chain.json")
    vocab = g["vocab"]
    V, gamma = len(vocab), len(g["drafts"])
    target = np.full((gamma + 1, V), -1.0)
    for i, top in enumerate(g["target_top1"]):
        target[i, vocab.index(top)] = 3.0
    target[gamma, :] = np.nan                          # the unspecified row
    drafts = np.array([vocab.index(t) for t in g["drafts"]])
    r = oracle.verify_greedy_sequence_early(target, drafts, gamma, gamma)
    assert r.status == oracle.SEQ_OK
    assert r.num_accepted == g["num_accepted"]
    assert [vocab[t] for t in r.tokens[: r.num_accepted + 1]] == g["committed"]
    assert r.rows_read == g["num_accepted"] + 1
    full = oracle.verify_greedy_sequence(target, drafts, gamma, gamma)
    assert full.status == oracle.SEQ_NONFINITE and full.num_accepted == -1


def test_wrblog_greedy_example_early():
    g = load_golden("wrblog_7_1_greedy.json")
    z = logits_of(g["p"])
    d = g["tokens"].index(g["draft"])
    r = oracle.verify_greedy_sequence_early(np.stack([z, z]), np.array([d]), 1, 1)
    assert r.num_accepted == g["num_accepted"]
    assert g["tokens"][r.tokens[0]] == g["emitted"]
    assert r.tokens[1] == -1
    assert r.rows_read == g["num_accepted"] + 1


@pytest.mark.parametrize("seed", range(40))
def test_matches_all_rows_greedy_on_valid_rows(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(2, 8))
    gmax = int(rng.integers(0, 6))
    gb = int(rng.integers(0, gmax + 1))
    target = rng.integers(-2, 3, size=(gmax + 1, V)).astype(np.float64)   # small ints: many ties
    argmax = [int(oracle.order_desc(target[i])[0]) for i in range(gmax + 1)]
    toks = np.array([argmax[i] if rng.random() < 0.6 else int(rng.integers(0, V)) for i in range(gmax)],
                    dtype=np.int64)
    e = oracle.verify_greedy_sequence_early(target, toks, gb, gmax)
    f = oracle.verify_greedy_sequence(target, toks, gb, gmax)
    assert e.status == f.status == oracle.SEQ_OK
    assert e.num_accepted == f.num_accepted
    assert np.array_equal(e.tokens, f.tokens)
    assert e.rows_read == e.num_accepted + 1


@pytest.mark.parametrize("bad", [np.nan, np.inf, "all_neg_inf"])
def test_row_errors_count_only_up_to_the_stop(bad):
    V, gmax = 5, 4
    target = np.tile(np.arange(V, dtype=np.float64), (gmax + 1, 1))     # argmax = V - 1 everywhere
    toks = np.array([V - 1, V - 1, 0, V - 1])                           # mismatch at position 2
    want = oracle.SEQ_EMPTY_SUPPORT if bad == "all_neg_inf" else oracle.SEQ_NONFINITE
    for row in range(gmax + 1):
        t = target.copy()
        if bad == "all_neg_inf":
            t[row, :] = -np.inf
        else:
            t[row, 1] = bad
        r = oracle.verify_greedy_sequence_early(t, toks, gmax, gmax)
        if row <= 2:
            assert r.status == want and r.num_accepted == -1 and r.rows_read == row + 1
            assert (r.tokens == -1).all()
        else:
            assert r.status == oracle.SEQ_OK and r.num_accepted == 2 and r.rows_read == 3
            assert list(r.tokens[:3]) == [V - 1, V - 1, V - 1]


def test_length_and_tokens_are_checked_before_any_row():
    target = np.full((3, 4), np.nan)
    r = oracle.verify_greedy_sequence_early(target, np.array([0, 7]), 2, 2)
    assert r.status == oracle.SEQ_BAD_TOKEN and r.rows_read == -1
    r = oracle.verify_greedy_sequence_early(target, np.array([0, 1]), 3, 2)
    assert r.status == oracle.SEQ_BAD_LENGTH


@pytest.mark.parametrize("gamma,a", [(1, 0.5), (4, 0.8), (6, 0.3), (8, 0.8)])
def test_rows_read_follow_the_truncated_geometric_law(gamma, a):
    """With each draft matching independently with probability a, the rows read
    equal the tokens emitted per round, whose mean is (1 - a^(gamma+1)) / (1 - a)
    [magicnet §4; rainlin §3].  Exact enumeration over the 2^gamma match patterns."""
    V = 3
    target = np.tile(np.array([0.0, 1.0, 0.5]), (gamma + 1, 1))        # argmax = 1 everywhere
    mean = 0.0
    for pattern in itertools.product([True, False], repeat=gamma):
        prob = np.prod([a if m else 1.0 - a for m in pattern])
        toks = np.array([1 if m else 2 for m in pattern], dtype=np.int64)
        r = oracle.verify_greedy_sequence_early(target, toks, gamma, gamma)
        mean += prob * r.rows_read
    assert abs(mean - (1.0 - a ** (gamma + 1)) / (1.0 - a)) < 1e-12
