"""GPU parity of sampling-mode draft-tree verification (spec_verify_sample_tree)
against the float64 oracle (its reading R17) [baisen §8; magicnet §7; wrblog §4-§6].

* random trees whose children are drawn independently from the draft
  distribution at their parent (the condition the method's law needs), both
  dtypes, two rule sets, ragged node counts: paths, counts and accepted tokens
  bit-exact and the drawn token under the CDF boundary rule, acceptance
  probabilities and residual mass within 1e-5 (the boundary rules of
  tests/helpers.py);
* the serving vocabulary (V = 128256, bf16, Zipf-shaped rows);
* a chain tree equals spec_verify_sample on the same rows bit for bit;
* data errors commit nothing in the documented order, a childless node's draft
  row is never read, unsupported requests are refused, the workspace is reusable.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_BOUNDARY, TOL_PROB, params_tuple, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_verification_44_gb300 import build
    build.build()


def make_sample_trees(B, N, V, dtype, seed, tp, dp, zipf=False):
    """Target rows, draft rows (target + noise), and trees whose node c carries a
    token drawn from the draft distribution at its parent (the oracle's q)."""
    from speculative_decoding_verification_44_gb300 import workloads
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    if zipf:
        tgt = workloads._zipf_rows(B * N, V, g, 0.5, "cpu").view(B, N, V)
    else:
        tgt = 2.0 * torch.randn(B, N, V, generator=g)
    dft = (tgt + 0.8 * torch.randn(B, N, V, generator=g)).to(dtype)
    tgt = tgt.to(dtype)
    q, _ = oracle.transform_rows(to_f64(dft).reshape(B * N, V), *params_tuple(dp))
    q = q.reshape(B, N, V)
    tokens = np.zeros((B, N), dtype=np.int32)
    parents = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        for c in range(1, N):
            p = int(rng.integers(0, c)) if rng.random() < 0.6 else c - 1
            parents[b, c] = p
            tokens[b, c] = int(rng.choice(V, p=q[b, p]))
    u_node = torch.from_numpy(rng.random((B, N)).astype(np.float32))
    u_sample = torch.from_numpy(rng.random(B).astype(np.float32))
    return tgt, dft, torch.from_numpy(tokens), torch.from_numpy(parents), u_node, u_sample


def gpu_tree(tgt, dft, tokens, parents, u_node, u_sample, tp, dp, nodes=None, workspace=None):
    import speculative_decoding_verification_44_gb300 as sv
    out, path = sv.verify_sample_tree(tgt.cuda(), dft.cuda(), tokens.cuda(), parents.cuda(), u_node.cuda(),
                                      u_sample.cuda(), tp, dp, None if nodes is None else nodes.cuda(),
                                      workspace=workspace)
    torch.cuda.synchronize()
    return out, path


def oracle_tree(tgt, dft, tokens, parents, u_node, u_sample, tp, dp, nodes=None):
    return oracle.verify_sample_tree(to_f64(tgt), to_f64(dft), tokens.numpy(), parents.numpy(),
                                     u_node.double().numpy(), u_sample.double().numpy(), params_tuple(tp),
                                     params_tuple(dp), None if nodes is None else nodes.numpy())


def compare_tree(out, path, ref, u_sample):
    toks = out.tokens.cpu().numpy()
    nacc = out.num_accepted.cpu().numpy()
    status = out.status.cpu().numpy()
    aprob = out.accept_prob.cpu().numpy()
    zres = out.residual_z.cpu().numpy()
    P = path.cpu().numpy()
    us = u_sample.double().numpy()
    c = dict(n=0, exact=0, flagged=0, boundary=0, errors=0, rejected=0, bonus=0)
    for b, r in enumerate(ref.seqs):
        c["n"] += 1
        if r.status & oracle.SEQ_ERROR_MASK:
            assert (status[b] & 0xFF) == (r.status & 0xFF), (b, status[b], r.status)
            assert nacc[b] == -1 and (toks[b] == -1).all() and (P[b] == -1).all(), b
            c["errors"] += 1
            continue
        assert (status[b] & 0xFF) == 0, (b, status[b])
        n = int(nacc[b])
        assert 0 <= toks[b, n] and (toks[b, n + 1:] == -1).all(), b
        if r.accept_margin < TOL_BOUNDARY or r.draft_ambiguous or toks[b, n] in r.sample_ambiguous \
                or r.tokens[r.num_accepted] in r.sample_ambiguous:
            c["flagged"] += 1
            continue
        assert n == r.num_accepted, (b, n, r.num_accepted)
        assert list(P[b, : n + 1]) == r.path and (P[b, n + 1:] == -1).all(), (b, P[b], r.path)
        assert (toks[b, :n] == r.tokens[:n]).all(), b
        tried = r.accept_prob >= 0
        np.testing.assert_allclose(aprob[b][tried], r.accept_prob[tried], atol=TOL_PROB, rtol=0,
                                   err_msg=f"accept_prob seq {b}")
        assert (aprob[b][~tried] == -1).all(), (b, aprob[b], r.accept_prob)
        assert (status[b] & 0x300) == (r.status & 0x300), (b, status[b], r.status)
        if r.residual_Z >= 0:
            c["rejected"] += 1
            assert abs(zres[b] - r.residual_Z) <= TOL_PROB, (b, zres[b], r.residual_Z)
        else:
            c["bonus"] += 1
            assert zres[b] == -1.0
        gt, ot = int(toks[b, n]), int(r.tokens[n])
        if gt == ot:
            c["exact"] += 1
        else:
            cdf, u = r.sample_cdf, us[b]
            ok = cdf[gt] >= u - TOL_BOUNDARY if gt < ot else cdf[gt - 1] <= u + TOL_BOUNDARY
            assert ok, (b, gt, ot, u)
            c["boundary"] += 1
    return c


RULES = [
    (dict(temperature=0.7, top_k=50, top_p=0.9), dict(temperature=0.7, top_k=50, top_p=0.9)),
    (dict(temperature=1.0, top_k=20, top_p=1.0), dict(temperature=1.3, top_k=40, top_p=0.95)),
    (dict(temperature=1.0, top_k=100, top_p=0.95), dict(temperature=0.9, top_k=120, top_p=1.0)),   # 4 chunks
    (dict(temperature=0.8, top_k=16, top_p=0.9), dict(temperature=0.8, top_k=32, top_p=0.9)),     # 1 chunk
]


@pytest.mark.parametrize("rules", range(len(RULES)))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_random_trees_match_the_oracle(rules, dtype):
    from speculative_decoding_verification_44_gb300 import SamplingParams
    tp, dp = SamplingParams(**RULES[rules][0]), SamplingParams(**RULES[rules][1])
    B, N, V = 24, 9, 4096
    x = make_sample_trees(B, N, V, dtype, 100 + rules, tp, dp)
    out, path = gpu_tree(*x, tp, dp)
    c = compare_tree(out, path, oracle_tree(*x, tp, dp), x[5])
    assert c["exact"] + c["boundary"] >= B - 2 and c["rejected"] > 0 and c["bonus"] > 0, c
    assert max(out.num_accepted.cpu().numpy()) >= 2, c             # some paths run past the root's children


def test_ragged_node_counts_and_wide_trees():
    from speculative_decoding_verification_44_gb300 import SamplingParams
    tp = dp = SamplingParams(0.8, 64, 0.95)
    B, N, V = 20, 32, 2048
    x = make_sample_trees(B, N, V, torch.bfloat16, 7, tp, dp)
    nodes = torch.from_numpy(np.random.default_rng(8).integers(1, N + 1, B).astype(np.int32))
    nodes[0] = 1                                                     # the root alone: a bonus draw
    out, path = gpu_tree(*x, tp, dp, nodes=nodes)
    c = compare_tree(out, path, oracle_tree(*x, tp, dp, nodes=nodes), x[5])
    assert c["exact"] + c["boundary"] >= B - 2, c
    assert out.num_accepted[0].item() == 0 and out.residual_z[0].item() == -1.0


def test_serving_vocabulary_zipf_rows():
    from speculative_decoding_verification_44_gb300 import SamplingParams
    tp = dp = SamplingParams(0.7, 50, 0.9)
    B, N, V = 8, 9, 128256
    x = make_sample_trees(B, N, V, torch.bfloat16, 21, tp, dp, zipf=True)
    out, path = gpu_tree(*x, tp, dp)
    c = compare_tree(out, path, oracle_tree(*x, tp, dp), x[5])
    assert c["exact"] + c["boundary"] + c["flagged"] == B and c["exact"] >= B - 2, c


def test_chain_tree_equals_the_linear_verifier():
    """One child per node: the same rows, uniforms and rules through spec_verify_sample."""
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import SamplingParams, workloads
    tp = dp = SamplingParams(0.7, 50, 0.9)
    for B, V, seed in [(16, 32768, 3), (64, 128256, 4)]:
        w = workloads.make(3, "cuda", draft_probs=lambda r, p: sv.transform_probs(r.contiguous(), p)[0],
                           B=B, V=V, replica=seed)
        G = w.G
        lin = sv.verify_sample(w.target_logits, w.draft_logits, w.draft_tokens, w.u_accept, w.u_sample, tp, dp)
        tokens = torch.cat([torch.zeros(B, 1, dtype=torch.int32, device="cuda"), w.draft_tokens.int()], dim=1)
        parents = torch.arange(-1, G, dtype=torch.int32, device="cuda").expand(B, G + 1).contiguous()
        dft = torch.cat([w.draft_logits, torch.zeros_like(w.draft_logits[:, :1])], dim=1).contiguous()
        u_node = torch.cat([torch.zeros(B, 1, device="cuda"), w.u_accept], dim=1).contiguous()
        tr, path = sv.verify_sample_tree(w.target_logits, dft, tokens.contiguous(), parents, u_node, w.u_sample,
                                         tp, dp)
        torch.cuda.synchronize()
        assert torch.equal(tr.num_accepted, lin.num_accepted)
        assert torch.equal(tr.tokens, lin.tokens)
        assert torch.equal(tr.status, lin.status)
        assert torch.equal(tr.residual_z, lin.residual_z)
        n = lin.num_accepted.cpu().numpy()
        la, ta = lin.accept_prob.cpu().numpy(), tr.accept_prob.cpu().numpy()
        for b in range(B):
            k = min(int(n[b]) + 1, G)                                 # positions the chain tried
            assert (ta[b, :k] == la[b, :k]).all(), b
            assert (ta[b, k:] == -1).all(), b
            assert list(path[b, : n[b] + 1].cpu().numpy()) == list(range(n[b] + 1))


def test_errors_commit_nothing_and_unread_rows():
    from speculative_decoding_verification_44_gb300 import SamplingParams
    tp = dp = SamplingParams(1.0, 30, 0.9)
    B, N, V = 8, 6, 1024
    tgt, dft, tokens, parents, u_node, u_sample = make_sample_trees(B, N, V, torch.float32, 5, tp, dp)
    parents[1, 3] = 3                                    # not an earlier node
    tokens[2, 4] = V                                     # out of range
    u_node[3, 2] = 1.0                                   # a uniform outside [0, 1)
    tgt[4, 5, 7] = float("nan")                          # a used target row
    childless = [c for c in range(1, N) if not (parents[5] == c).any()]
    dft[5, childless[0], 9] = float("nan")               # a childless node's draft row: not read
    with_child = int(parents[6, 1:].max())
    dft[6, with_child, 3] = float("inf")                 # a draft row that is read
    nodes = torch.full((B,), N, dtype=torch.int32)
    nodes[7] = N + 1                                     # a bad node count
    x = (tgt, dft, tokens, parents, u_node, u_sample)
    out, path = gpu_tree(*x, tp, dp, nodes=nodes)
    ref = oracle_tree(*x, tp, dp, nodes=nodes)
    compare_tree(out, path, ref, u_sample)
    st = out.status.cpu().numpy() & 0xFF
    assert list(st[1:8]) == [oracle.SEQ_BAD_TREE, oracle.SEQ_BAD_TOKEN, oracle.SEQ_BAD_UNIFORM,
                             oracle.SEQ_NONFINITE, 0, oracle.SEQ_NONFINITE, oracle.SEQ_BAD_LENGTH]


def test_unsupported_requests_are_refused():
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import SamplingParams, _lib
    x = make_sample_trees(2, 4, 512, torch.float32, 1, SamplingParams(1.0, 10, 1.0), SamplingParams(1.0, 10, 1.0))
    for tp in [SamplingParams(1.0, 0, 0.9), SamplingParams(1.0, 200, 1.0)]:      # full-row rules
        with pytest.raises(_lib.SpecError) as e:
            gpu_tree(*x, tp, tp)
        assert e.value.status == _lib.SPEC_ERR_UNSUPPORTED
    with pytest.raises(_lib.SpecError) as e:
        sv.tree_sample_workspace_size(2, 33, 512, SamplingParams(1.0, 10, 1.0), SamplingParams(1.0, 10, 1.0))
    assert e.value.status == _lib.SPEC_ERR_UNSUPPORTED


def test_workspace_is_reusable():
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import SamplingParams
    tp = dp = SamplingParams(0.9, 32, 0.95)
    x = make_sample_trees(12, 8, 3000, torch.bfloat16, 9, tp, dp)
    ws = sv.new_workspace(sv.tree_sample_workspace_size(12, 8, 3000, tp, dp), "cuda")
    a, pa = gpu_tree(*x, tp, dp, workspace=ws)
    b, pb = gpu_tree(*x, tp, dp, workspace=ws)
    for f in ("tokens", "num_accepted", "status", "accept_prob", "residual_z"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    assert torch.equal(pa, pb)
