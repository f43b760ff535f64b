"""Oracle pins for greedy draft-tree verification (reading R15 of the oracle).

The pages say a tree of candidate paths is verified in one forward and the
best path is accepted [baisen §8; magicnet §7];
greedy verification of a tree is then pinned by:

* a chain tree (every node's parent is the node before it) is exactly the
  linear greedy verifier [wrblog §7.1];
* brute force: with distinct sibling tokens the accepted node is the deepest
  node whose whole root path agrees with the target's argmaxes;
* losslessness: with a deterministic tabular target, the emitted tokens are
  the target's own greedy continuation of the prefix;
* the error order: length, node tokens, parents, rows.
"""
import numpy as np
import pytest

import oracle


def random_tree(rng, n, V, distinct=True):
    parents = np.zeros(n, dtype=np.int64)
    tokens = np.zeros(n, dtype=np.int64)
    used = {0: set()}
    for i in range(1, n):
        while True:
            p = int(rng.integers(0, i))
            free = [t for t in range(V) if t not in used[p]] if distinct else list(range(V))
            if free:
                break
        parents[i] = p
        tokens[i] = int(rng.choice(free))
        used[p].add(int(tokens[i]))
        used[i] = set()
    return tokens, parents


def test_chain_tree_is_linear_greedy():
    rng = np.random.default_rng(1)
    for trial in range(200):
        G, V = int(rng.integers(0, 7)), int(rng.integers(2, 9))
        target = rng.normal(0.0, 1.0, (G + 1, V)).round(1)      # rounding makes ties common
        d = rng.integers(0, V, G)
        for i in range(G):                                     # often the argmax: long prefixes
            if rng.random() < 0.6:
                d[i] = int(np.argmax(target[i]))
        lin = oracle.verify_greedy_sequence(target, d, G, G)
        tokens = np.concatenate([[0], d])
        parents = np.arange(-1, G)
        tree = oracle.verify_greedy_tree_sequence(target, tokens, parents, G + 1, G + 1)
        assert tree.num_accepted == lin.num_accepted and tree.status == lin.status
        np.testing.assert_array_equal(tree.tokens, lin.tokens)
        assert tree.path == list(range(lin.num_accepted + 1))


def test_deepest_matching_node_by_brute_force():
    rng = np.random.default_rng(2)
    for trial in range(300):
        n, V = int(rng.integers(1, 14)), int(rng.integers(2, 6))
        tokens, parents = random_tree(rng, n, V)
        target = rng.normal(0.0, 1.0, (n, V))
        g = np.argmax(target, axis=1)
        for i in range(1, n):                                  # make many edges match
            if rng.random() < 0.5:
                sib = [c for c in range(1, n) if parents[c] == parents[i] and c != i]
                if int(g[parents[i]]) not in [int(tokens[c]) for c in sib]:
                    tokens[i] = g[parents[i]]
        # a node matches when every edge on its root path carries the parent's argmax
        def depth_if_matching(i):
            dpt = 0
            while i != 0:
                if tokens[i] != g[parents[i]]:
                    return -1
                i, dpt = int(parents[i]), dpt + 1
            return dpt
        depths = [depth_if_matching(i) for i in range(n)]
        best = int(np.argmax(depths))
        res = oracle.verify_greedy_tree_sequence(target, tokens, parents, n, n)
        assert res.path[-1] == best and res.num_accepted == depths[best]
        assert res.tokens[res.num_accepted] == g[best]


def test_emits_the_target_greedy_continuation():
    V = 5
    rng = np.random.default_rng(3)
    table = {}

    def logits(prefix):
        if prefix not in table:
            table[prefix] = rng.normal(0.0, 1.0, V)
        return table[prefix]

    def greedy_continuation(prefix, n):
        out = []
        for _ in range(n):
            t = int(np.argmax(logits(prefix + tuple(out))))
            out.append(t)
        return out

    for trial in range(200):
        n = int(rng.integers(1, 12))
        tokens, parents = random_tree(rng, n, V)
        root = tuple(int(x) for x in rng.integers(0, V, int(rng.integers(0, 3))))
        paths = [root]
        for i in range(1, n):
            paths.append(paths[parents[i]] + (int(tokens[i]),))
        # steer some nodes onto the target's own choice
        for i in range(1, n):
            want = int(np.argmax(logits(paths[parents[i]])))
            sib = [int(tokens[c]) for c in range(1, n) if parents[c] == parents[i] and c != i]
            if rng.random() < 0.6 and want not in sib:
                tokens[i] = want
                paths[i] = paths[parents[i]] + (want,)
                for c in range(i + 1, n):                       # descendants follow the new prefix
                    paths[c] = paths[parents[c]] + (int(tokens[c]),)
        target = np.stack([logits(p) for p in paths])
        res = oracle.verify_greedy_tree_sequence(target, tokens, parents, n, n)
        L = res.num_accepted
        assert list(res.tokens[: L + 1]) == greedy_continuation(root, L + 1)
        assert (res.tokens[L + 1:] == -1).all()


def test_error_order():
    V, n = 6, 5
    target = np.zeros((n, V))
    tokens = np.array([0, 1, 2, 3, 4])
    parents = np.array([-1, 0, 1, 1, 2])
    ok = oracle.verify_greedy_tree_sequence(target, tokens, parents, n, n)
    assert ok.status == oracle.SEQ_OK
    assert oracle.verify_greedy_tree_sequence(target, tokens, parents, 0, n).status == oracle.SEQ_BAD_LENGTH
    assert oracle.verify_greedy_tree_sequence(target, tokens, parents, n + 1, n).status == oracle.SEQ_BAD_LENGTH
    bad_tok = tokens.copy(); bad_tok[3] = V
    bad_par = parents.copy(); bad_par[2] = 2
    both = bad_par.copy()
    assert oracle.verify_greedy_tree_sequence(target, bad_tok, both, n, n).status == oracle.SEQ_BAD_TOKEN
    assert oracle.verify_greedy_tree_sequence(target, tokens, bad_par, n, n).status == oracle.SEQ_BAD_TREE
    nan_row = target.copy(); nan_row[4, 2] = np.nan
    assert oracle.verify_greedy_tree_sequence(nan_row, tokens, bad_par, n, n).status == oracle.SEQ_BAD_TREE
    assert oracle.verify_greedy_tree_sequence(nan_row, tokens, parents, n, n).status == oracle.SEQ_NONFINITE
    # nodes beyond n are never read
    assert oracle.verify_greedy_tree_sequence(nan_row, tokens, parents, 4, n).status == oracle.SEQ_OK
