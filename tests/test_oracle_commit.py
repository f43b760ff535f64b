"""Oracle pins for per-sequence sampling rules and the end-of-sequence commit.

* End-of-sequence commit [wrblog §14.3]: no token is committed after the EOS.
  - Exact law: with rounds repeated until L tokens or an EOS, the law of the
    committed sequence equals the target's autoregressive law stopped at the
    EOS (enumeration over drafts and uniform intervals, V <= 4, gamma <= 2) --
    speculative decoding stays lossless with the cut [wrblog §6.1].
  - Invariants on random batches: the committed block is a prefix of the
    uncut one; the EOS is its last token; blocks without an EOS are unchanged.
* Per-sequence rules [wrblog §15]: a batch whose sequences carry their own
  temperature / top-k / top-p gives each sequence the result of verifying it
  alone under its rules; a rule outside its domain fails only its sequence,
  after the length, token and uniform checks.
"""
import functools

import numpy as np
import pytest

import oracle

T1 = (1.0, 0, 1.0)


def logits_of(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, dtype=np.float64))


def round_law_eos(p_of, q_of, prefix, V, gamma, eos):
    """Law of the block one verification round commits from ``prefix``, EOS cut applied."""
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
        probe = oracle.verify_sample_sequence(target, draft, toks, np.zeros(gamma), 0.5, T1, T1,
                                              gamma, gamma, False)
        a = probe.accept_prob[:gamma]
        for j in range(gamma + 1):
            if j < gamma:
                w_acc = np.prod(a[:j]) * (1.0 - a[j])
                u_acc = np.array([a[i] / 2 for i in range(j)] + [(1.0 + a[j]) / 2] + [0.5] * (gamma - j - 1))
            else:
                w_acc = np.prod(a)
                u_acc = a / 2
            if w_acc == 0.0:
                continue
            res = oracle.verify_sample_sequence(target, draft, toks, u_acc, 0.5, T1, T1, gamma, gamma,
                                                False, keep_cdf=True)
            cdf = res.sample_cdf
            lo = np.concatenate([[0.0], cdf[:-1]])
            for x in range(V):
                width = cdf[x] - lo[x]
                if width <= 0:
                    continue
                r = oracle.verify_sample_sequence(target, draft, toks, u_acc, (lo[x] + cdf[x]) / 2,
                                                  T1, T1, gamma, gamma, False)
                r = oracle.commit_at_eos(r, eos)
                block = tuple(int(t) for t in r.tokens if t >= 0)
                assert len(block) == r.num_emitted
                law[block] = law.get(block, 0.0) + w_d * w_acc * width
    return law


@pytest.mark.parametrize("V,gamma,L,seed", [(3, 1, 3, 1), (3, 2, 3, 2), (4, 2, 3, 3), (4, 1, 4, 4)])
def test_eos_cut_keeps_the_target_law(V, gamma, L, seed):
    rng = np.random.default_rng(seed)
    eos = V - 1
    tables_p, tables_q = {}, {}

    def dist(table, ctx):
        if ctx not in table:
            table[ctx] = rng.dirichlet(np.ones(V))
        return table[ctx]

    p_of = functools.partial(dist, tables_p)
    q_of = functools.partial(dist, tables_q)

    @functools.lru_cache(maxsize=None)
    def law_from(prefix):
        if len(prefix) >= L or (prefix and prefix[-1] == eos):
            return {prefix[:L]: 1.0}
        out = {}
        for block, w in round_law_eos(p_of, q_of, prefix, V, gamma, eos).items():
            assert eos not in block[:-1]                       # nothing after the EOS
            for seq, w2 in law_from(prefix + block).items():
                out[seq] = out.get(seq, 0.0) + w * w2
        return out

    got = law_from(())

    def target_law(prefix):
        if len(prefix) >= L or (prefix and prefix[-1] == eos):
            return {prefix[:L]: 1.0}
        out = {}
        p = p_of(prefix)
        for x in range(V):
            for seq, w in target_law(prefix + (x,)).items():
                out[seq] = out.get(seq, 0.0) + p[x] * w
        return out

    want = target_law(())
    assert set(got) == set(want)
    for k in want:
        assert abs(got[k] - want[k]) < 1e-12, (k, got[k], want[k])


def random_batch(rng, B=40, G=4, V=12):
    target = rng.normal(0.0, 1.5, (B, G + 1, V))
    draft = target[:, :G] + rng.normal(0.0, 0.7, (B, G, V))
    tokens = rng.integers(0, V, (B, G))
    tokens[:, 0] = np.argmax(target[:, 0], axis=1)        # the first draft is often accepted
    ua, us = rng.random((B, G)), rng.random(B)
    gam = rng.integers(0, G + 1, B)
    onehot = rng.random(B) < 0.25
    return target, draft, tokens, ua, us, gam, onehot


def test_eos_commit_invariants():
    rng = np.random.default_rng(5)
    target, draft, tokens, ua, us, gam, onehot = random_batch(rng)
    base = oracle.verify_sample(target, draft, tokens, ua, us, T1, T1, gam, onehot)
    cuts = 0
    for eos in range(12):
        cut = oracle.verify_sample(target, draft, tokens, ua, us, T1, T1, gam, onehot, eos_token=eos)
        for b, (r0, r1) in enumerate(zip(base.seqs, cut.seqs)):
            blk0 = [int(t) for t in r0.tokens if t >= 0]
            blk1 = [int(t) for t in r1.tokens if t >= 0]
            assert blk1 == blk0[: len(blk1)]                     # a prefix of the uncut block
            assert len(blk1) == r1.num_emitted
            if eos in blk0:
                assert blk1[-1] == eos and eos not in blk1[:-1]
                assert r1.status & oracle.SEQ_FLAG_EOS
                cuts += len(blk1) < len(blk0)
                if len(blk1) < len(blk0):                         # cut at an accepted draft
                    assert r1.num_accepted == len(blk1) and r1.num_accepted <= r0.num_accepted
            else:
                assert blk1 == blk0 and r1.num_accepted == r0.num_accepted
                assert not r1.status & oracle.SEQ_FLAG_EOS
            np.testing.assert_array_equal(r1.accept_prob, r0.accept_prob)
    assert cuts > 5


def test_per_sequence_rules_equal_single_sequence_calls():
    rng = np.random.default_rng(7)
    target, draft, tokens, ua, us, gam, onehot = random_batch(rng, B=24)
    rules = [(1.0, 0, 1.0), (0.7, 3, 0.9), (1.3, 0, 0.8), (0.5, 1, 1.0), (2.0, 5, 0.6)]
    per = [(rules[b % 5], rules[(b + 2) % 5]) for b in range(24)]
    got = oracle.verify_sample(target, draft, tokens, ua, us, T1, T1, gam, onehot, params_per_seq=per)
    for b in range(24):
        alone = oracle.verify_sample(target[b:b + 1], draft[b:b + 1], tokens[b:b + 1], ua[b:b + 1], us[b:b + 1],
                                     per[b][0], per[b][1], gam[b:b + 1], onehot[b:b + 1])
        np.testing.assert_array_equal(got.tokens[b], alone.tokens[0])
        assert got.num_accepted[b] == alone.num_accepted[0] and got.status[b] == alone.status[0]
    same = oracle.verify_sample(target, draft, tokens, ua, us, T1, T1, gam, onehot,
                                params_per_seq=[(T1, T1)] * 24)
    base = oracle.verify_sample(target, draft, tokens, ua, us, T1, T1, gam, onehot)
    np.testing.assert_array_equal(same.tokens, base.tokens)
    np.testing.assert_array_equal(same.accept_prob, base.accept_prob)


def test_bad_rules_fail_only_their_sequence():
    rng = np.random.default_rng(9)
    target, draft, tokens, ua, us, gam, onehot = random_batch(rng, B=8)
    gam[:] = 3
    onehot[:] = False
    onehot[6] = True
    bad = [(0.0, 0, 1.0), (float("nan"), 0, 1.0), (1.0, -1, 1.0), (1.0, 0, 0.0), (1.0, 0, 1.5)]
    per = [(T1, T1)] * 8
    per = [(bad[0], T1), (T1, bad[1]), (bad[2], T1), (T1, bad[3]), (bad[4], bad[4]), (T1, T1),
           (T1, bad[0]), (T1, T1)]
    us = us.copy()
    us[5] = 1.0                                        # a bad uniform is reported before a bad rule
    per[5] = (bad[0], T1)
    r = oracle.verify_sample(target, draft, tokens, ua, us, T1, T1, gam, onehot, params_per_seq=per)
    st = [int(s) & oracle.SEQ_ERROR_MASK for s in r.status]
    assert st[:6] == [oracle.SEQ_BAD_PARAMS] * 5 + [oracle.SEQ_BAD_UNIFORM]
    assert st[6] == oracle.SEQ_OK                      # one-hot: its draft rule is not used
    assert st[7] == oracle.SEQ_OK
    assert (r.num_accepted[:6] == -1).all()
