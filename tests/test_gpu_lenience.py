"""GPU parity of lenient verification [magicnet §8] (spec_verify_sample_lenient).

* lenience = 1 reproduces spec_verify_sample bit for bit;
* for lenience < 1 the outputs match the float64 oracle under the same
  boundary rules as the lossless path (tests/helpers.py), on every row path:
  streaming top-k lists, full rows with and without top-p, one-hot drafts;
* over many rounds with fixed logits the first emitted token follows the
  oracle's exact lenient law (chi-square), which respects the 1/beta bound.
"""
import numpy as np
import pytest
import scipy.stats
import torch

import oracle
from helpers import check_sample_counts, gpu_sample, oracle_probs, params_tuple, run_oracle_sample, to_f64
from test_oracle_lenience import first_token_law

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_verification_44_gb300 import build
    build.build()


def workload(wid, **kw):
    from speculative_decoding_verification_44_gb300 import workloads
    return workloads.make(wid, "cpu", draft_probs=oracle_probs, **kw).to("cuda")


CASES = [(1, dict(B=2000)), (2, dict()), (3, dict(B=12, V=20000)), (5, dict(B=24, V=30000))]


@pytest.mark.parametrize("wid,kw", CASES[2:])
def test_lenience_one_is_the_plain_call(wid, kw):
    w = workload(wid, **kw)
    a = gpu_sample(w)
    b = gpu_sample(w, lenience=1.0)
    torch.cuda.synchronize()
    for name in ("tokens", "num_accepted", "status", "accept_prob", "residual_z"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


@pytest.mark.parametrize("beta", [0.9, 0.5, 0.1])
@pytest.mark.parametrize("wid,kw", CASES)
def test_lenient_matches_oracle(wid, kw, beta):
    w = workload(wid, **kw)
    out = gpu_sample(w, lenience=beta)
    torch.cuda.synchronize()
    c = check_sample_counts(out, run_oracle_sample(w, lenience=float(np.float32(beta))), w)
    if wid == 1 and beta == 0.9:
        assert c["rejected"] > 50 and c["bonus"] > 50
    if beta == 0.1:
        assert c["bonus"] >= c["rejected"]          # loose acceptance: most rounds accept all


def test_invalid_lenience_is_refused():
    from speculative_decoding_verification_44_gb300 import _lib
    w = workload(3, B=2, V=4096)
    for bad in (0.0, -0.25, 1.5, float("nan"), float("inf")):
        with pytest.raises(_lib.SpecError) as e:
            gpu_sample(w, lenience=bad)
        assert e.value.status == 1


@pytest.mark.parametrize("beta", [0.5, 0.2])
def test_lenient_first_token_law(beta):
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import workloads
    rounds = 400_000
    base = workloads.make(1, "cpu", draft_probs=oracle_probs)
    G, V = base.G, base.V
    tp = params_tuple(base.target_params)
    p = oracle.transform_row(to_f64(base.target_logits[0, 0]), *tp).probs
    q = oracle.transform_row(to_f64(base.draft_logits[0, 0]), *tp).probs
    law, _ = first_token_law(p, q, float(np.float32(beta)))
    assert np.all(law <= p / float(np.float32(beta)) + 1e-12)
    rng = np.random.default_rng(int(beta * 1000))
    qs = [oracle.transform_row(to_f64(base.draft_logits[0, i]), *tp).probs for i in range(G)]
    drafts = np.stack([rng.choice(V, size=rounds, p=qi / qi.sum()) for qi in qs], axis=1)
    g = torch.Generator(device="cuda").manual_seed(7)
    out = sv.verify_sample(base.target_logits.expand(rounds, -1, -1).contiguous().cuda(),
                           base.draft_logits.expand(rounds, -1, -1).contiguous().cuda(),
                           torch.from_numpy(drafts).to(torch.int32).cuda(),
                           torch.rand(rounds, G, generator=g, device="cuda"),
                           torch.rand(rounds, generator=g, device="cuda"),
                           base.target_params, base.draft_params, lenience=beta)
    torch.cuda.synchronize()
    assert (out.status.cpu().numpy() & 0xFF == 0).all()
    first = out.tokens[:, 0].cpu().numpy()
    counts = np.bincount(first, minlength=V)
    expect = law * rounds
    keep = expect > 5
    chi2, pval = scipy.stats.chisquare(counts[keep], expect[keep] * counts[keep].sum() / expect[keep].sum())
    assert pval > 1e-6, (chi2, pval)
    assert counts[~keep].sum() <= max(50, 10 * expect[~keep].sum())
