"""GPU parity of greedy draft-tree verification (spec_verify_greedy_tree)
against the float64 oracle [baisen §8; magicnet §7]: bit-exact paths, tokens
and counts.

* chain trees reproduce spec_verify_greedy on the same rows;
* random trees (a third of the nodes steered onto their parent's argmax, so
  paths run deep) at several vocabulary sizes, both dtypes, ragged node counts;
* data errors (length, node token, parent, non-finite row) commit nothing,
  nodes past a sequence's count are never read, the workspace is reusable.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_verification_44_gb300 import build
    build.build()


def make_trees(B, N, V, dtype, seed, steer=0.35):
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    logits = (2.0 * torch.randn(B, N, V, generator=g)).to(dtype)
    arg = to_f64(logits).argmax(axis=2)                     # the lowest index wins ties
    tokens = np.zeros((B, N), dtype=np.int32)
    parents = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        for i in range(1, N):
            p = int(rng.integers(0, i)) if rng.random() < 0.7 else i - 1
            parents[b, i] = p
            tokens[b, i] = int(arg[b, p]) if rng.random() < steer else int(rng.integers(0, V))
    return logits, torch.from_numpy(tokens), torch.from_numpy(parents)


def check(logits, tokens, parents, nodes=None):
    import speculative_decoding_verification_44_gb300 as sv
    out, path = sv.verify_greedy_tree(logits.cuda(), tokens.cuda(), parents.cuda(),
                                      None if nodes is None else nodes.cuda())
    torch.cuda.synchronize()
    ref = oracle.verify_greedy_tree(to_f64(logits), tokens.numpy(), parents.numpy(),
                                    None if nodes is None else nodes.numpy())
    np.testing.assert_array_equal(out.num_accepted.cpu().numpy(), ref.num_accepted)
    np.testing.assert_array_equal(out.tokens.cpu().numpy(), ref.tokens)
    np.testing.assert_array_equal(out.status.cpu().numpy(), ref.status)
    P = path.cpu().numpy()
    for b, r in enumerate(ref.seqs):
        if r.num_accepted >= 0:
            assert list(P[b, : r.num_accepted + 1]) == r.path and (P[b, r.num_accepted + 1:] == -1).all()
        else:
            assert (P[b] == -1).all()
    return ref


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V", [4099, 32000])
def test_random_trees_match_oracle(dtype, V):
    logits, tokens, parents = make_trees(24, 16, V, dtype, seed=V + (dtype == torch.float32))
    ref = check(logits, tokens, parents)
    assert ref.num_accepted.max() >= 3                      # some paths run deep


def test_ragged_node_counts_and_reuse():
    import speculative_decoding_verification_44_gb300 as sv
    logits, tokens, parents = make_trees(20, 12, 8192, torch.bfloat16, seed=7, steer=0.5)
    nodes = torch.from_numpy(np.random.default_rng(8).integers(1, 13, 20).astype(np.int32))
    logits[:, -1, 5] = float("nan")                         # read only by sequences with 12 nodes
    ws = sv.new_workspace(sv.tree_workspace_size(20, 12), "cuda")
    for _ in range(2):                                      # the workspace is left reusable
        out, _ = sv.verify_greedy_tree(logits.cuda(), tokens.cuda(), parents.cuda(), nodes.cuda(), workspace=ws)
    torch.cuda.synchronize()
    ref = check(logits, tokens, parents, nodes)
    np.testing.assert_array_equal(out.tokens.cpu().numpy(), ref.tokens)
    full = nodes.numpy() == 12
    assert ((out.status.cpu().numpy() == oracle.SEQ_NONFINITE) == full).all()


def test_chain_trees_are_spec_verify_greedy():
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import workloads
    w = workloads.make(4, "cpu", B=32, V=20000)
    B, G = w.B, w.G
    tokens = torch.cat([torch.zeros(B, 1, dtype=torch.int32), w.draft_tokens.to(torch.int32)], dim=1)
    parents = torch.arange(-1, G, dtype=torch.int32).expand(B, G + 1).contiguous()
    tree, path = sv.verify_greedy_tree(w.target_logits.cuda(), tokens.cuda(), parents.cuda())
    lin = sv.verify_greedy(w.target_logits.cuda(), w.draft_tokens.cuda())
    torch.cuda.synchronize()
    assert torch.equal(tree.tokens, lin.tokens) and torch.equal(tree.num_accepted, lin.num_accepted)
    assert torch.equal(tree.status, lin.status)


def test_data_errors_commit_nothing():
    logits, tokens, parents = make_trees(6, 8, 3000, torch.bfloat16, seed=11)
    nodes = torch.tensor([8, 0, 9, 8, 8, 8], dtype=torch.int32)   # 0 and 9: bad lengths
    tokens[3, 4] = 3000                                             # bad token
    parents[4, 5] = 5                                               # not an earlier node
    logits[5, 2, 7] = float("inf")                                  # non-finite row
    ref = check(logits, tokens, parents, nodes)
    assert [int(s) for s in ref.status] == [0, 1, 1, 2, 7, 4]
