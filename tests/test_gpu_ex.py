"""GPU parity of spec_verify_sample_ex: per-sequence sampling rules [wrblog §15]
and the end-of-sequence commit [wrblog §14.3].

* default options, and per-sequence rules that repeat the scalar ones,
  reproduce spec_verify_sample bit for bit (the device prepares each rule with
  the host's arithmetic);
* mixed per-sequence rules (kept-list and full-row paths in one launch, each
  side its own rules) match the float64 oracle under the usual boundary rules;
* with an end-of-sequence token the committed blocks, counts and the EOS flag
  match the oracle's commit, on the kept-list path and the full-row path (whose
  draw runs in the second kernel);
* a per-sequence rule outside its domain fails only its sequence.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_sample_counts, gpu_sample, oracle_probs, run_oracle_sample

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


def same(a, b, names=("tokens", "num_accepted", "status", "accept_prob", "residual_z")):
    for n in names:
        assert torch.equal(getattr(a, n), getattr(b, n)), n


@pytest.mark.parametrize("wid,kw", [(1, dict(B=300)), (3, dict(B=12, V=20000)), (5, dict(B=24, V=30000))])
def test_defaults_and_repeated_rules_are_the_plain_call(wid, kw):
    w = workload(wid, **kw)
    plain = gpu_sample(w)
    ex = gpu_sample(w, eos_token=-1)
    per = gpu_sample(w, target_rules=[w.target_params] * w.B, draft_rules=[w.draft_params] * w.B)
    torch.cuda.synchronize()
    same(plain, ex)
    same(plain, per)
    ok = plain.num_accepted >= 0
    assert torch.equal(ex.num_emitted[ok], plain.num_accepted[ok] + 1)


RULES = [(0.7, 50, 0.9), (1.0, 0, 0.95), (1.3, 0, 1.0), (0.8, 128, 0.8), (1.0, 1, 1.0), (0.6, 7, 1.0)]


@pytest.mark.parametrize("V", [9000, 20001])
def test_mixed_rules_match_oracle(V):
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300.workloads import sample_from_probs
    w = workload(3, B=18, V=V)
    tr = [sv.SamplingParams(*RULES[b % len(RULES)]) for b in range(w.B)]
    dr = [sv.SamplingParams(*RULES[(b + 2) % len(RULES)]) for b in range(w.B)]
    # draft tokens drawn from each sequence's own q
    rows = []
    for b in range(w.B):
        q = oracle_probs(w.draft_logits[b].cpu(), dr[b])
        rows.append(sample_from_probs(q, torch.Generator().manual_seed(100 + b)))
    w.draft_tokens = torch.stack(rows).to(torch.int32).cuda()
    out = gpu_sample(w, target_rules=tr, draft_rules=dr)
    torch.cuda.synchronize()
    c = check_sample_counts(out, run_oracle_sample(w, rules=list(zip(tr, dr))), w)
    assert c["errors"] == 0 and c["n"] == w.B


@pytest.mark.parametrize("wid,kw", [(3, dict(B=16, V=12000)), (5, dict(B=24, V=30000)), (1, dict(B=400))])
def test_eos_commit_matches_oracle(wid, kw):
    w = workload(wid, **kw)
    # make the EOS the clear favourite of target and draft at position 1 in half the
    # sequences and draft it there, so that blocks get cut at an accepted EOS draft
    eos = 3
    toks = w.draft_tokens.cpu().clone()
    tl, dl = w.target_logits.cpu().clone(), w.draft_logits.cpu().clone()
    tl[::2, 1, eos] = tl[::2, 1].max(dim=-1).values + 12.0
    dl[::2, 1, eos] = dl[::2, 1].max(dim=-1).values + 12.0
    toks[::2, 1] = eos
    w.target_logits, w.draft_logits, w.draft_tokens = tl.cuda(), dl.cuda(), toks.cuda()
    out = gpu_sample(w, eos_token=eos)
    torch.cuda.synchronize()
    ref = run_oracle_sample(w, eos_token=eos)
    c = check_sample_counts(out, ref, w)
    nem = out.num_emitted.cpu().numpy()
    st = out.status.cpu().numpy()
    cut = 0
    for b, r in enumerate(ref.seqs):
        if r.status & oracle.SEQ_ERROR_MASK:
            continue
        if r.accept_margin < 1e-6 or r.draft_ambiguous:
            continue
        assert nem[b] == r.num_emitted, (b, nem[b], r.num_emitted)
        if r.num_emitted == r.num_accepted:          # cut at an accepted EOS draft
            cut += 1
            assert st[b] & oracle.SEQ_FLAG_EOS
            assert out.residual_z[b].item() == -1.0
    assert cut > 0 and c["n"] == w.B


def test_bad_rules_fail_only_their_sequence():
    import speculative_decoding_verification_44_gb300 as sv
    w = workload(3, B=8, V=4096)
    good = w.target_params
    tr = [good] * 8
    dr = [w.draft_params] * 8
    tr[1] = sv.SamplingParams(0.0, 50, 0.9)
    tr[3] = sv.SamplingParams(float("nan"), 50, 0.9)
    dr[5] = sv.SamplingParams(1.0, -3, 0.9)
    dr[6] = sv.SamplingParams(1.0, 50, 1.5)
    out = gpu_sample(w, target_rules=tr, draft_rules=dr)
    torch.cuda.synchronize()
    st = [s & 0xFF for s in out.status.tolist()]
    assert [st[i] for i in (1, 3, 5, 6)] == [6, 6, 6, 6]
    assert [st[i] for i in (0, 2, 4, 7)] == [0, 0, 0, 0]
    assert (out.num_accepted.cpu()[[1, 3, 5, 6]] == -1).all()
    assert (out.num_emitted.cpu()[[1, 3, 5, 6]] == -1).all()


def test_kept_list_promise():
    """kept_list_only: the same results as without the promise when every rule keeps
    it; a per-sequence rule that breaks it fails only its sequence; scalar rules
    that break it are refused before launch."""
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import _lib
    w = workload(3, B=10, V=9000)
    kept = [(0.7, 50, 0.9), (1.0, 1, 1.0), (0.9, 128, 0.8), (1.2, 7, 1.0)]
    tr = [sv.SamplingParams(*kept[b % 4]) for b in range(w.B)]
    dr = [sv.SamplingParams(*kept[(b + 1) % 4]) for b in range(w.B)]
    a = gpu_sample(w, target_rules=tr, draft_rules=dr)
    b = gpu_sample(w, target_rules=tr, draft_rules=dr, kept_list_only=True)
    torch.cuda.synchronize()
    same(a, b)
    tr[3] = sv.SamplingParams(1.0, 0, 0.9)            # top-k off: the full-row path
    dr[6] = sv.SamplingParams(1.0, 300, 1.0)          # top-k above the kept-list limit
    c = gpu_sample(w, target_rules=tr, draft_rules=dr, kept_list_only=True)
    torch.cuda.synchronize()
    st = [s & 0xFF for s in c.status.tolist()]
    assert st[3] == 6 and st[6] == 6 and all(st[i] == 0 for i in range(w.B) if i not in (3, 6))
    w.target_params = sv.SamplingParams(1.0, 0, 0.9)
    with pytest.raises(_lib.SpecError) as e:
        gpu_sample(w, target_rules=tr, draft_rules=dr, kept_list_only=True,
                   workspace=sv.new_workspace(1 << 24, "cuda"))
    assert e.value.status == 1
