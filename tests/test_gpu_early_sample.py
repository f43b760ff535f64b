"""GPU parity of early-exit sampling verification (spec_verify_sample_ex with
early_exit): the sequential verifier of [wrblog §6], positions read in order,
each sequence stopping at its first failed row or rejected draft.

* on valid rows the outputs equal the all-rows call bit for bit (tokens,
  counts, status, residual mass), with a_i up to the stop and -1 after it;
* against the float64 oracle's early-exit reading under the usual boundary
  rules, on both row paths and both dtypes, with one-hot drafts and ragged
  lengths;
* NaN rows after each sequence's stop do not fail it, whether or not the
  launch happened to skip them (several waves of row CTAs, so most are
  skipped), while the all-rows call fails those sequences;
* the workspace stays reusable: early and all-rows calls alternate on one
  workspace with the same results.
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


def same_up_to_stop(early, full):
    for n in ("tokens", "num_accepted", "status", "residual_z"):
        assert torch.equal(getattr(early, n), getattr(full, n)), n
    j = full.num_accepted.cpu().numpy()
    ae, af = early.accept_prob.cpu().numpy(), full.accept_prob.cpu().numpy()
    for b in range(len(j)):
        if j[b] < 0:
            continue
        np.testing.assert_array_equal(ae[b, : j[b] + 1], af[b, : j[b] + 1])   # a_i up to the stop
        assert (ae[b, j[b] + 1:] == -1).all(), b


CASES = [(1, dict(B=300)), (2, dict(B=8)), (3, dict(B=12, V=20000)), (5, dict(B=24, V=30000)),
         (5, dict(B=96, V=4099))]


@pytest.mark.parametrize("wid,kw", CASES)
def test_early_equals_all_rows_on_valid_rows(wid, kw):
    w = workload(wid, **kw)
    full = gpu_sample(w, eos_token=-1)
    early = gpu_sample(w, early_exit=True)
    torch.cuda.synchronize()
    same_up_to_stop(early, full)


@pytest.mark.parametrize("wid,kw", CASES)
def test_early_matches_oracle(wid, kw):
    w = workload(wid, **kw)
    out = gpu_sample(w, early_exit=True)
    torch.cuda.synchronize()
    check_sample_counts(out, run_oracle_sample(w, early_exit=True), w, early=True)


@pytest.mark.parametrize("V", [30000, 4099])
def test_rows_after_the_stop_do_not_fail_the_sequence(V):
    """Several waves of row CTAs (512 sequences of up to 7 drafts): NaN in every
    row after each sequence's stop.  The early call returns the clean all-rows
    result; the all-rows call fails exactly the sequences that stopped early."""
    w = workload(5, B=512, V=V)
    clean = gpu_sample(w, eos_token=-1)
    torch.cuda.synchronize()
    j = clean.num_accepted.cpu().numpy()
    gam = w.gamma_per_seq.cpu().numpy()
    onehot = w.draft_is_onehot.cpu().numpy().astype(bool)
    tl, dl = w.target_logits.clone(), w.draft_logits.clone()
    poisoned = []
    for b in range(w.B):
        if 0 <= j[b] < gam[b]:
            tl[b, j[b] + 1:] = float("nan")
            if not onehot[b]:
                dl[b, j[b] + 1:] = float("nan")
            poisoned.append(b)
    assert len(poisoned) > w.B // 4
    w.target_logits, w.draft_logits = tl, dl
    early = gpu_sample(w, early_exit=True)
    again = gpu_sample(w, early_exit=True)
    full = gpu_sample(w, eos_token=-1)
    torch.cuda.synchronize()
    same_up_to_stop(early, clean)
    same_up_to_stop(again, clean)
    st = full.status.cpu().numpy() & 0xFF
    assert (st[poisoned] == oracle.SEQ_NONFINITE).all()
    rest = np.setdiff1d(np.arange(w.B), poisoned)
    assert (st[rest] == (clean.status.cpu().numpy()[rest] & 0xFF)).all()


def test_failed_row_before_the_stop_fails_the_sequence():
    """NaN in the target row of each sequence's stop position (a row the early
    verifier must read): the same failure as the oracle's."""
    w = workload(5, B=64, V=4099)
    clean = gpu_sample(w, eos_token=-1)
    torch.cuda.synchronize()
    j = clean.num_accepted.cpu().numpy()
    tl = w.target_logits.clone()
    for b in range(w.B):
        if j[b] >= 0:
            tl[b, j[b], 5] = float("nan")
    w.target_logits = tl
    out = gpu_sample(w, early_exit=True)
    torch.cuda.synchronize()
    ref = run_oracle_sample(w, early_exit=True)
    st = out.status.cpu().numpy()
    for b in range(w.B):
        assert st[b] == ref.status[b], (b, st[b], ref.status[b])
        if j[b] >= 0:
            assert st[b] & 0xFF == oracle.SEQ_NONFINITE


def test_workspace_reuse_across_modes():
    import speculative_decoding_verification_44_gb300 as sv
    w = workload(5, B=200, V=4099)
    ws = sv.new_workspace(sv.workspace_size(w.B, w.G, w.V, w.target_params, w.draft_params), "cuda")
    first = gpu_sample(w, workspace=ws, early_exit=True)
    full = gpu_sample(w, workspace=ws, eos_token=-1)
    second = gpu_sample(w, workspace=ws, early_exit=True)
    torch.cuda.synchronize()
    same_up_to_stop(first, full)
    same_up_to_stop(second, full)


@pytest.mark.parametrize("V", [9000, 30000])
def test_early_exit_with_rules_and_eos(V):
    """Early exit together with the other options: per-sequence rules (both row
    paths in one launch) and an end-of-sequence commit, against the oracle's
    early-exit reading with the same rules and the same EOS cut."""
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300.workloads import sample_from_probs
    rules = [(0.7, 50, 0.9), (1.0, 0, 0.95), (1.3, 0, 1.0), (0.8, 128, 0.8), (0.6, 7, 1.0)]
    w = workload(5, B=40, V=V)
    tr = [sv.SamplingParams(*rules[b % len(rules)]) for b in range(w.B)]
    dr = [sv.SamplingParams(*rules[(b + 2) % len(rules)]) for b in range(w.B)]
    toks = []
    for b in range(w.B):
        q = oracle_probs(w.draft_logits[b].cpu(), dr[b])
        toks.append(sample_from_probs(q, torch.Generator().manual_seed(300 + b)))
    w.draft_tokens = torch.stack(toks).to(torch.int32).cuda()
    eos = int(w.draft_tokens[0, 0])
    out = gpu_sample(w, target_rules=tr, draft_rules=dr, eos_token=eos, early_exit=True)
    torch.cuda.synchronize()
    ref = run_oracle_sample(w, rules=list(zip(tr, dr)), eos_token=eos, early_exit=True)
    c = check_sample_counts(out, ref, w, early=True)
    assert c["errors"] == 0 and c["n"] == w.B
    nem = out.num_emitted.cpu().numpy()
    for b, r in enumerate(ref.seqs):
        if r.accept_margin >= 1e-6 and not r.draft_ambiguous:
            assert nem[b] == r.num_emitted, (b, nem[b], r.num_emitted)
