"""Pins of the oracle's sampling-mode tree verification (reading R17 of the oracle).

The pages say a draft tree is verified in one forward and the best path is
accepted [baisen §8; magicnet §7], but give no sampling rule; what they do fix
is that speculative sampling keeps the target's distribution [wrblog §5.1,
§6.1; rainlin §2].  So the pins are:

* Exact output law: with each node's children drawn independently from the
  draft distribution at that node, the law of the emitted tokens over repeated
  rounds equals the target's autoregressive law, for several tree shapes, by
  exhaustive enumeration of node tokens, acceptance decisions and the final
  draw on a 3-token vocabulary.  The decisions are enumerated through the
  oracle's own trace of tried nodes and acceptance probabilities, so the law is
  the oracle's, not a retyped algorithm.
* A chain (one child per node) is the linear verifier exactly.
* Closed-form consequences: a sibling that repeats a rejected token is never
  accepted; a root without children draws the bonus from p; error order.
"""
import functools
import itertools

import numpy as np
import pytest

import oracle

T1 = (1.0, 0, 1.0)


def logits_of(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, dtype=np.float64))


def tables(V, seed, zero_frac=0.25):
    """Random tabular target / draft next-token models p(.|ctx), q(.|ctx)."""
    rng = np.random.default_rng(seed)
    cache = {}

    def dist(kind, ctx):
        key = (kind, ctx)
        if key not in cache:
            r = np.random.default_rng(abs(hash((seed, kind, ctx))) % (2 ** 32))
            x = r.dirichlet(np.ones(V))
            mask = r.random(V) < zero_frac
            if mask.all():
                mask[r.integers(V)] = False
            x = np.where(mask, 0.0, x)
            cache[key] = x / x.sum()
        return cache[key]
    del rng
    return (lambda ctx: dist("p", ctx)), (lambda ctx: dist("q", ctx))


def path_to(v, parents, tokens):
    out = []
    while v > 0:
        out.append(int(tokens[v]))
        v = int(parents[v])
    return tuple(reversed(out))


def tree_round_law(p_of, q_of, prefix, V, parents):
    """Law of the block one tree round emits from context ``prefix`` (tree shape ``parents``)."""
    n = len(parents)
    parents = np.array(parents, dtype=np.int64)
    law = {}
    for toks in itertools.product(range(V), repeat=n - 1):
        tokens = np.array((0,) + toks, dtype=np.int64)
        w_tok = 1.0
        for c in range(1, n):
            w_tok *= q_of(prefix + path_to(int(parents[c]), parents, tokens))[tokens[c]]
        if w_tok == 0.0:
            continue
        ctx = [prefix + path_to(v, parents, tokens) for v in range(n)]
        target = np.stack([logits_of(p_of(c)) for c in ctx])
        draft = np.stack([logits_of(q_of(c)) for c in ctx])

        def run(assign, us):
            u_node = np.array([assign.get(c, 0.0) for c in range(n)])
            return oracle.verify_sample_tree_sequence(target, draft, tokens, parents, u_node, us, n, n, T1, T1)

        def explore(assign, w):
            probe = run(assign, 0.5)
            assert probe.status & oracle.SEQ_ERROR_MASK == oracle.SEQ_OK
            for c, a_c in probe.tree_trace:
                if c not in assign:
                    if a_c > 0:
                        explore({**assign, c: a_c / 2}, w * a_c)
                    if a_c < 1:
                        explore({**assign, c: (1.0 + a_c) / 2}, w * (1.0 - a_c))
                    return
            cdf = probe.sample_cdf
            lo = np.concatenate([[0.0], cdf[:-1]])
            for x in range(V):
                width = cdf[x] - lo[x]
                if width <= 0:
                    continue
                r = run(assign, (lo[x] + cdf[x]) / 2)
                L = r.num_accepted
                assert r.tokens[L] == x and [tuple(t for t, _ in r.tree_trace)] == [tuple(t for t, _ in probe.tree_trace)]
                block = tuple(int(t) for t in r.tokens[: L + 1])
                law[block] = law.get(block, 0.0) + w_tok * w * width

        explore({}, 1.0)
    return law


def sequence_law(round_law, L):
    @functools.lru_cache(maxsize=None)
    def law_from(prefix):
        if len(prefix) >= L:
            return {prefix[:L]: 1.0}
        out = {}
        for block, w in round_law(prefix).items():
            for seq, w2 in law_from(prefix + block).items():
                out[seq] = out.get(seq, 0.0) + w * w2
        return out
    return law_from(())


def target_law(p_of, V, L):
    out = {}
    for seq in itertools.product(range(V), repeat=L):
        pr = 1.0
        for t in range(L):
            pr *= p_of(seq[:t])[seq[t]]
        if pr > 0:
            out[seq] = pr
    return out


SHAPES = [
    [-1, 0, 0],            # two children of the root
    [-1, 0, 0, 0],         # three children
    [-1, 0, 0, 1],         # two children, the first with a child of its own
    [-1, 0, 1, 1],         # one child, then two grandchildren
    [-1, 0, 1],            # a chain
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("seed", [1, 2])
def test_tree_round_keeps_the_target_law(shape, seed):
    V, L = 3, 3
    p_of, q_of = tables(V, seed)
    law = sequence_law(lambda prefix: tree_round_law(p_of, q_of, prefix, V, shape), L)
    ref = target_law(p_of, V, L)
    assert set(k for k, v in law.items() if v > 1e-15) == set(ref)
    for k, v in ref.items():
        assert abs(law.get(k, 0.0) - v) < 1e-12, (k, law.get(k), v)


@pytest.mark.parametrize("shape", SHAPES)
def test_first_token_follows_p_root(shape):
    V = 3
    p_of, q_of = tables(V, 7, zero_frac=0.0)
    law = tree_round_law(p_of, q_of, (), V, shape)
    first = np.zeros(V)
    for block, w in law.items():
        first[block[0]] += w
    np.testing.assert_allclose(first, p_of(()), atol=1e-12)


def test_law_fails_for_a_residual_that_is_not_updated():
    """The enumeration catches the plausible mistake of trying every child against p
    itself (no residual update): the emitted law then differs from the target's."""
    V = 3
    p_of, q_of = tables(V, 3, zero_frac=0.0)
    shape = np.array([-1, 0, 0])
    law = {}
    for toks in itertools.product(range(V), repeat=2):
        q = q_of(())
        w_tok = q[toks[0]] * q[toks[1]]
        p = p_of(())
        # wrong rule: each child against p, residual (p - q)+ only at the end
        a1 = min(1.0, p[toks[0]] / q[toks[0]])
        a2 = min(1.0, p[toks[1]] / q[toks[1]])
        res = np.maximum(p - q, 0.0)
        res = res / res.sum()
        first = np.zeros(V)
        first[toks[0]] += a1
        first[toks[1]] += (1 - a1) * a2
        first += (1 - a1) * (1 - a2) * res
        for x in range(V):
            law[x] = law.get(x, 0.0) + w_tok * first[x]
    assert max(abs(law[x] - p_of(())[x]) for x in range(V)) > 1e-3
    # while the oracle's rule keeps p
    ok = tree_round_law(p_of, q_of, (), V, list(shape))
    first = np.zeros(V)
    for block, w in ok.items():
        first[block[0]] += w
    np.testing.assert_allclose(first, p_of(()), atol=1e-12)


def test_chain_tree_is_the_linear_verifier():
    rng = np.random.default_rng(11)
    for trial in range(40):
        V = int(rng.integers(8, 200))
        G = int(rng.integers(1, 6))
        tgt = rng.normal(0, 2, (G + 1, V))
        dft = tgt[:G] + rng.normal(0, 1, (G, V))
        params = [(1.0, 0, 1.0), (0.7, 5, 0.9), (1.3, 0, 0.8)][trial % 3]
        q = [oracle.transform_row(dft[i], *params).probs for i in range(G)]
        d = np.array([rng.choice(V, p=q[i]) for i in range(G)])
        ua = rng.random(G)
        us = float(rng.random())
        lin = oracle.verify_sample_sequence(tgt, dft, d, ua, us, params, params, G, G, False)
        tokens = np.concatenate([[0], d])
        parents = np.arange(-1, G)
        draft_rows = np.concatenate([dft, np.zeros((1, V))])
        u_node = np.concatenate([[0.0], ua])
        tr = oracle.verify_sample_tree_sequence(tgt, draft_rows, tokens, parents, u_node, us, G + 1, G + 1,
                                                params, params)
        assert tr.status == lin.status
        assert tr.num_accepted == lin.num_accepted
        assert (tr.tokens == lin.tokens).all()
        assert tr.residual_Z == lin.residual_Z
        tried = lin.num_accepted + (1 if lin.num_accepted < G else 0)
        np.testing.assert_array_equal(tr.accept_prob[:tried], lin.accept_prob[:tried])
        assert tr.path == list(range(lin.num_accepted + 1))


def test_repeated_rejected_token_is_never_accepted():
    """Rejecting token x leaves r(x) = (p(x) - q(x))+ / Z = 0 (a rejection needs
    p(x) < q(x)), so a sibling repeating x has acceptance probability 0."""
    V = 5
    rng = np.random.default_rng(5)
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    x = int(np.argmax(q / p))                       # p(x) < q(x): rejectable
    assert p[x] < q[x]
    tgt = np.stack([logits_of(p)] + [logits_of(p)] * 2)
    dft = np.stack([logits_of(q)] + [logits_of(q)] * 2)
    tokens = np.array([0, x, x])
    parents = np.array([-1, 0, 0])
    a1 = p[x] / q[x]
    res = oracle.verify_sample_tree_sequence(tgt, dft, tokens, parents, np.array([0.0, (1 + a1) / 2, 0.0]),
                                             0.3, 3, 3, T1, T1)
    assert [c for c, _ in res.tree_trace] == [1, 2]
    assert res.tree_trace[1][1] == 0.0 and res.num_accepted == 0
    assert res.tokens[0] != x                       # drawn from (p - q)+, where x has no mass


def test_root_without_children_draws_the_bonus_from_p():
    V = 6
    p = np.array([0.1, 0.2, 0.3, 0.1, 0.2, 0.1])
    tgt = logits_of(p)[None, :]
    res = oracle.verify_sample_tree_sequence(tgt, np.zeros((1, V)), np.array([0]), np.array([-1]),
                                             np.array([0.0]), 0.35, 1, 1, T1, T1)
    assert res.num_accepted == 0 and res.tokens[0] == 2 and res.residual_Z == -1.0   # cumsum .1 .3 .6


def test_error_order_and_unused_rows():
    V, n = 8, 4
    rng = np.random.default_rng(2)
    tgt = rng.normal(0, 1, (n, V))
    dft = rng.normal(0, 1, (n, V))
    tokens = np.array([0, 1, 2, 3])
    parents = np.array([-1, 0, 0, 1])
    u = np.array([0.0, 0.5, 0.5, 0.5])
    run = lambda **kw: oracle.verify_sample_tree_sequence(
        kw.get("tgt", tgt), kw.get("dft", dft), kw.get("tokens", tokens), kw.get("parents", parents),
        kw.get("u", u), kw.get("us", 0.5), kw.get("n", n), n, T1, T1)
    assert run(n=0).status == oracle.SEQ_BAD_LENGTH
    assert run(tokens=np.array([0, 1, V, 3]), parents=np.array([-1, 0, 5, 1])).status == oracle.SEQ_BAD_TOKEN
    assert run(parents=np.array([-1, 0, 2, 1])).status == oracle.SEQ_BAD_TREE
    assert run(u=np.array([0.0, 0.5, 1.0, 0.5])).status == oracle.SEQ_BAD_UNIFORM
    bad = tgt.copy()
    bad[3, 2] = np.nan
    assert run(tgt=bad).status == oracle.SEQ_NONFINITE          # every node's target row is read
    leaf_draft = dft.copy()
    leaf_draft[2, 0] = np.nan                                    # node 2 has no children: not read
    assert run(dft=leaf_draft).status & oracle.SEQ_ERROR_MASK == oracle.SEQ_OK
    parent_draft = dft.copy()
    parent_draft[1, 0] = np.nan                                  # node 1 has a child: read
    assert run(dft=parent_draft).status == oracle.SEQ_NONFINITE
