"""Pins for the early-exit sampling oracle (reading R16).

The sequential verifier of [wrblog §6] reads position after position and
stops at the first draft the target rejects.  These tests pin the early-exit
oracle to the page example of [baisen §4], to the all-rows sampling oracle on
valid inputs (whose law is pinned elsewhere), and to its error semantics:
rows after the stop are never read, rows up to it are.
"""
import numpy as np
import pytest

import oracle
from conftest import load_golden


def logits_of(p):
    return np.log(np.asarray(p, dtype=np.float64))


OFF = (1.0, 0, 1.0)   # temperature 1, no top-k, no top-p: p and q are the rows' softmax


def one(target, draft, tokens, u_acc, u_s, g, gmax, early, tp=OFF, dp=OFF, one_hot=False, lenience=1.0):
    return oracle.verify_sample_sequence(target, draft, np.asarray(tokens), np.asarray(u_acc, dtype=np.float64),
                                         u_s, tp, dp, g, gmax, one_hot, lenience=lenience, early_exit=early)


def test_baisen_rejection_never_reads_the_bonus_row():
    """[baisen §4]: with u = 0.9 > a = 5/6 "mat" is rejected and "sat" comes
    from the residual.  The sequential verifier stops there, so the bonus row
    may hold NaN; the all-rows verifier fails on it."""
    g = load_golden("baisen_4_mat_sat_ran.json")
    p, q = logits_of(g["p"]), logits_of(g["q"])
    d = g["tokens"].index(g["draft"])
    target = np.stack([p, np.full_like(p, np.nan)])
    r = one(target, q[None, :], [d], [0.9], 0.77, 1, 1, early=True)
    assert r.status == oracle.SEQ_OK and r.num_accepted == 0 and r.rows_read == 1
    assert g["tokens"][r.tokens[0]] == "sat"
    assert abs(r.accept_prob[0] - g["accept_probability_exact"]) < 1e-12
    full = one(target, q[None, :], [d], [0.9], 0.77, 1, 1, early=False)
    assert full.status == oracle.SEQ_NONFINITE and full.num_accepted == -1
    # accepted (u = 0 < a): the bonus row is read and fails the sequence in both
    acc = one(target, q[None, :], [d], [0.0], 0.77, 1, 1, early=True)
    assert acc.status == oracle.SEQ_NONFINITE and acc.rows_read == 2


def random_case(rng, V, gmax):
    target = rng.normal(0.0, 2.0, (gmax + 1, V))
    draft = target[:gmax] + rng.normal(0.0, 1.0, (gmax, V))
    tokens = rng.integers(0, V, gmax)
    u_acc = rng.random(gmax)
    return target, draft, tokens, u_acc, float(rng.random())


RULES = [(OFF, OFF), ((0.7, 3, 0.9), (1.3, 0, 0.8)), ((1.0, 0, 0.5), (0.5, 2, 1.0))]


@pytest.mark.parametrize("seed", range(36))
def test_matches_all_rows_on_valid_rows(seed):
    """Valid rows: the same tokens, counts, flags and residual mass as the
    all-rows oracle; a_i up to the stop, -1 after it; rows read = stop + 1."""
    rng = np.random.default_rng(seed)
    V, gmax = int(rng.integers(2, 9)), int(rng.integers(0, 6))
    gb = int(rng.integers(0, gmax + 1))
    target, draft, tokens, u_acc, u_s = random_case(rng, V, gmax)
    tp, dp = RULES[seed % len(RULES)]
    one_hot = seed % 4 == 3
    lenience = (1.0, 0.5)[seed % 2]
    full = one(target, draft, tokens, u_acc, u_s, gb, gmax, False, tp, dp, one_hot, lenience)
    early = one(target, draft, tokens, u_acc, u_s, gb, gmax, True, tp, dp, one_hot, lenience)
    assert full.status == early.status
    np.testing.assert_array_equal(full.tokens, early.tokens)
    assert full.num_accepted == early.num_accepted
    assert full.residual_Z == early.residual_Z
    j = full.num_accepted
    assert early.rows_read == j + 1
    np.testing.assert_array_equal(early.accept_prob[: min(j + 1, gb)], full.accept_prob[: min(j + 1, gb)])
    assert (early.accept_prob[j + 1:] == -1.0).all()
    assert early.accept_margin == full.accept_margin


@pytest.mark.parametrize("seed", range(24))
def test_rows_after_the_stop_are_never_read(seed):
    """NaN in the first target row after the stop (and in every later row):
    the early result equals the all-rows result on the clean rows, while the
    all-rows verifier fails.  Placing the NaN at stop + 1 catches a verifier
    that reads one row too many."""
    rng = np.random.default_rng(100 + seed)
    V, gmax = int(rng.integers(3, 9)), int(rng.integers(2, 6))
    target, draft, tokens, u_acc, u_s = random_case(rng, V, gmax)
    # a sure rejection no later than position k: a draft token with q > p there
    # (so a_k < 1) and u_k just below 1
    k = int(rng.integers(0, gmax))
    sm = lambda z: np.exp(z - z.max()) / np.exp(z - z.max()).sum()
    tokens[k] = int(np.argmax(sm(draft[k]) - sm(target[k])))
    u_acc[k] = np.nextafter(1.0, 0.0)
    full = one(target, draft, tokens, u_acc, u_s, gmax, gmax, False)
    j = full.num_accepted
    assert j <= k
    bad_t, bad_d = target.copy(), draft.copy()
    bad_t[j + 1:] = np.nan
    bad_d[j + 1:] = np.nan
    early = one(bad_t, bad_d, tokens, u_acc, u_s, gmax, gmax, True)
    assert early.status == full.status and early.num_accepted == j and early.rows_read == j + 1
    np.testing.assert_array_equal(early.tokens, full.tokens)
    assert one(bad_t, bad_d, tokens, u_acc, u_s, gmax, gmax, False).status == oracle.SEQ_NONFINITE


@pytest.mark.parametrize("which", ["target", "draft"])
def test_a_failed_row_up_to_the_stop_fails_the_sequence(which):
    """Position 0 is accepted (u = 0), position 1 rejected (u just below 1 and
    a_1 < 1): a NaN in target row 1 or draft row 1 is read and fails the
    sequence; rows read = 2."""
    rng = np.random.default_rng(7)
    V, gmax = 6, 3
    target, draft, tokens, u_acc, u_s = random_case(rng, V, gmax)
    sm = lambda z: np.exp(z - z.max()) / np.exp(z - z.max()).sum()
    tokens[1] = int(np.argmax(sm(draft[1]) - sm(target[1])))   # q > p there: a_1 < 1
    u_acc[0] = 0.0
    u_acc[1] = np.nextafter(1.0, 0.0)
    clean = one(target, draft, tokens, u_acc, u_s, gmax, gmax, True)
    assert clean.num_accepted == 1 and clean.rows_read == 2
    (target if which == "target" else draft)[1, 2] = np.nan
    r = one(target, draft, tokens, u_acc, u_s, gmax, gmax, True)
    assert r.status == oracle.SEQ_NONFINITE and r.num_accepted == -1 and r.rows_read == 2


def test_input_checks_come_first():
    """Lengths, tokens, uniforms and rules are checked before any row, as in
    the all-rows verifier."""
    rng = np.random.default_rng(3)
    target, draft, tokens, u_acc, u_s = random_case(rng, 5, 3)
    target[:] = np.nan
    assert one(target, draft, [0, 9, 0], u_acc, u_s, 3, 3, True).status == oracle.SEQ_BAD_TOKEN
    assert one(target, draft, tokens, [0.1, 1.0, 0.2], u_s, 3, 3, True).status == oracle.SEQ_BAD_UNIFORM
    assert one(target, draft, tokens, u_acc, u_s, 3, 3, True, tp=(0.0, 0, 1.0)).status == oracle.SEQ_BAD_PARAMS
    assert one(target, draft, tokens, u_acc, u_s, 4, 3, True).status == oracle.SEQ_BAD_LENGTH


def test_batch_wrapper_passes_the_flag():
    rng = np.random.default_rng(11)
    B, gmax, V = 5, 3, 7
    target = rng.normal(0, 2, (B, gmax + 1, V))
    draft = target[:, :gmax] + rng.normal(0, 1, (B, gmax, V))
    tokens = rng.integers(0, V, (B, gmax))
    u_acc, u_s = rng.random((B, gmax)), rng.random(B)
    full = oracle.verify_sample(target, draft, tokens, u_acc, u_s, OFF, OFF)
    target[:, gmax] = np.nan                      # the bonus rows
    early = oracle.verify_sample(target, draft, tokens, u_acc, u_s, OFF, OFF, early_exit=True)
    for b in range(B):
        if full.num_accepted[b] < gmax:
            assert early.status[b] == full.status[b] and early.num_accepted[b] == full.num_accepted[b]
        else:
            assert early.status[b] == oracle.SEQ_NONFINITE


def test_target_row_is_checked_before_its_draft_row():
    """R16's order within a position: target row i, then draft row i.  Target row
    1 all -inf (empty support) and draft row 1 NaN: the target's failure is the
    one reported."""
    rng = np.random.default_rng(21)
    target, draft, tokens, u_acc, u_s = random_case(rng, 6, 3)
    u_acc[0] = 0.0                                   # position 0 accepted: position 1 is read
    target[1] = -np.inf
    draft[1, 0] = np.nan
    r = one(target, draft, tokens, u_acc, u_s, 3, 3, True)
    assert r.status == oracle.SEQ_EMPTY_SUPPORT and r.rows_read == 2


@pytest.mark.parametrize("seed", range(12))
def test_eos_commit_and_per_sequence_rules_under_early_exit(seed):
    """The end-of-sequence cut (R14) and per-sequence rules (R13) apply to the
    early-exit result exactly as to the all-rows one: on valid rows the
    committed blocks agree."""
    rng = np.random.default_rng(500 + seed)
    B, gmax, V = 6, 4, 7
    target = rng.normal(0, 2, (B, gmax + 1, V))
    draft = target[:, :gmax] + rng.normal(0, 1, (B, gmax, V))
    tokens = rng.integers(0, V, (B, gmax))
    u_acc, u_s = rng.random((B, gmax)), rng.random(B)
    per = [RULES[(b + seed) % len(RULES)] for b in range(B)]
    eos = int(tokens[0, 0])
    kw = dict(params_per_seq=per, eos_token=eos, lenience=(1.0, 0.7)[seed % 2])
    full = oracle.verify_sample(target, draft, tokens, u_acc, u_s, OFF, OFF, **kw)
    early = oracle.verify_sample(target, draft, tokens, u_acc, u_s, OFF, OFF, early_exit=True, **kw)
    np.testing.assert_array_equal(full.tokens, early.tokens)
    np.testing.assert_array_equal(full.num_accepted, early.num_accepted)
    np.testing.assert_array_equal(full.status, early.status)
    assert [r.num_emitted for r in full.seqs] == [r.num_emitted for r in early.seqs]
