"""Statistics of the GPU path over 10^6 rounds with fixed logits (workload 1 shape).

Draft tokens are drawn from the oracle's q, uniforms are fresh per round.
Checks [wrblog §14.1; rainlin §2]:
* the first emitted token follows p_1; given i accepted drafts, the token at
  position i+1 follows p_{i+1} (chi-square, and total-variation distance);
* per-position empirical acceptance matches sum_x min(p_i, q_i);
* the histogram of accepted counts matches the exact truncated law
  P(A = k) = prod_{i<k} a_i (1 - a_k), P(A = gamma) = prod a_i.
"""
import numpy as np
import pytest
import scipy.stats
import torch

import oracle
from helpers import oracle_probs, params_tuple, to_f64

pytestmark = pytest.mark.gpu

ROUNDS = 1_000_000


@pytest.fixture(scope="module")
def run():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import build, workloads
    build.build()
    base = workloads.make(1, "cpu", draft_probs=oracle_probs)
    G, V = base.G, base.V
    tp = params_tuple(base.target_params)
    p = np.stack([oracle.transform_row(to_f64(base.target_logits[0, i]), *tp).probs for i in range(G + 1)])
    q = np.stack([oracle.transform_row(to_f64(base.draft_logits[0, i]), *tp).probs for i in range(G)])
    rng = np.random.default_rng(12345)
    drafts = np.stack([rng.choice(V, size=ROUNDS, p=q[i] / q[i].sum()) for i in range(G)], axis=1)
    tl = base.target_logits.expand(ROUNDS, -1, -1).contiguous().cuda()
    dl = base.draft_logits.expand(ROUNDS, -1, -1).contiguous().cuda()
    g = torch.Generator(device="cuda").manual_seed(99)
    ua = torch.rand(ROUNDS, G, generator=g, device="cuda")
    us = torch.rand(ROUNDS, generator=g, device="cuda")
    out = sv.verify_sample(tl, dl, torch.from_numpy(drafts).to(torch.int32).cuda(), ua, us,
                           base.target_params, base.draft_params)
    torch.cuda.synchronize()
    return dict(p=p, q=q, G=G, V=V, drafts=drafts, tokens=out.tokens.cpu().numpy(),
                nacc=out.num_accepted.cpu().numpy(), status=out.status.cpu().numpy())


def test_no_errors(run):
    assert (run["status"] & 0xFF == 0).all()


@pytest.mark.parametrize("pos", [0, 1, 2, 3, 4])
def test_emitted_token_follows_target(run, pos):
    sel = run["nacc"] >= pos
    toks = run["tokens"][sel, pos]
    n = toks.size
    assert n > 20_000
    counts = np.bincount(toks, minlength=run["V"])
    expect = run["p"][pos] * n
    keep = expect > 5
    chi2, pval = scipy.stats.chisquare(counts[keep], expect[keep] * counts[keep].sum() / expect[keep].sum())
    assert pval > 1e-6, (pos, chi2, pval)
    tv = 0.5 * np.abs(counts / n - run["p"][pos]).sum()
    assert tv < 3.0 * np.sqrt(run["V"] / n), tv
    assert counts[~keep].sum() <= max(50, 10 * expect[~keep].sum())


def test_per_position_acceptance_and_count_law(run):
    G = run["G"]
    alpha = np.array([oracle.acceptance_rate(run["p"][i], run["q"][i]) for i in range(G)])
    nacc = run["nacc"]
    for i in range(G):
        reached = nacc >= i
        acc = (nacc[reached] > i).mean()
        n = reached.sum()
        assert abs(acc - alpha[i]) < 5 * np.sqrt(alpha[i] * (1 - alpha[i]) / n), (i, acc, alpha[i])
    law = np.array([np.prod(alpha[:k]) * (1 - alpha[k]) for k in range(G)] + [np.prod(alpha)])
    counts = np.bincount(nacc, minlength=G + 1)
    chi2, pval = scipy.stats.chisquare(counts, law * counts.sum())
    assert pval > 1e-6, (counts, law, pval)


def test_accepted_prefix_is_the_drafts(run):
    toks, nacc, d = run["tokens"], run["nacc"], run["drafts"]
    for k in range(1, run["G"] + 1):
        sel = nacc >= k
        assert (toks[sel, :k] == d[sel, :k]).all()
    cols = np.arange(toks.shape[1])[None, :]
    assert (toks[cols > nacc[:, None]] == -1).all()
