"""Parity at the full workload sizes, in the launch configuration the benchmark
times (one launch over the whole batch), on sequences the oracle recomputes
one by one.  Inputs are generated on the GPU and copied to the host; draft
tokens are drawn from the oracle's q."""
import numpy as np
import pytest
import torch

from helpers import (compare_greedy, compare_sample, gpu_greedy, gpu_sample, oracle_probs,
                     run_oracle_greedy, run_oracle_sample)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_verification_44_gb300 import build
    build.build()


def make(wid):
    from speculative_decoding_verification_44_gb300 import workloads
    return workloads.make(wid, "cuda", draft_probs=oracle_probs)


def test_serving_shape_full_batch():
    """B=64, gamma=5, V=128256 bf16, T=0.7, top-k 50, top-p 0.9: all 64 sequences."""
    w = make(3)
    out = gpu_sample(w)
    torch.cuda.synchronize()
    c = compare_sample(out, run_oracle_sample(w), w)
    assert c["n"] == 64 and c["flagged"] + c["boundary"] <= 3, c


def test_greedy_full_batch_sampled():
    """B=256, gamma=8, V=152064 bf16: 64 sequences spread over the batch."""
    w = make(4)
    out = gpu_greedy(w)
    torch.cuda.synchronize()
    seqs = list(range(0, 256, 4))
    assert compare_greedy(out, run_oracle_greedy(w, seqs), w, seqs) == 64
    # batch-wide invariants at any size
    nacc = out.num_accepted.cpu().numpy()
    toks = out.tokens.cpu().numpy()
    d = w.draft_tokens.cpu().numpy()
    assert ((nacc >= 0) & (nacc <= 8)).all()
    for b in range(256):
        assert (toks[b, : nacc[b]] == d[b, : nacc[b]]).all()
    am = w.target_logits.float().argmax(dim=2).cpu().numpy()
    assert (toks[np.arange(256), nacc] == am[np.arange(256), nacc]).mean() > 0.99   # ties are rare


def test_ragged_mixed_full_batch_sampled():
    """B=512, gamma_b in 1..7, V=256000 bf16, top-p 0.95; model-like and one-hot drafts."""
    w = make(5)
    out = gpu_sample(w)
    torch.cuda.synchronize()
    seqs = list(range(0, 512, 16)) + list(range(7, 512, 32))
    c = compare_sample(out, run_oracle_sample(w, seqs), w, seqs)
    assert c["n"] == len(seqs) and c["flagged"] + c["boundary"] <= 3, c
    assert (out.status.cpu() & 0xFF == 0).all()


def test_serving_full_batch_lenient_and_per_sequence_rules():
    """The serving workload through spec_verify_sample_lenient (beta 0.5) and through
    spec_verify_sample_ex with the workload's rule given per sequence (kept-list
    promise, as the benchmark runs it) and an end-of-sequence token: all 64 sequences."""
    import oracle
    w = make(3)
    len_out = gpu_sample(w, lenience=0.5)
    torch.cuda.synchronize()
    c = compare_sample(len_out, run_oracle_sample(w, lenience=float(np.float32(0.5))), w)
    assert c["n"] == 64 and c["flagged"] + c["boundary"] <= 3, c
    eos = int(w.draft_tokens[0, 0])
    ex = gpu_sample(w, eos_token=eos, target_rules=[w.target_params] * 64, draft_rules=[w.draft_params] * 64,
                    kept_list_only=True)
    torch.cuda.synchronize()
    ref = run_oracle_sample(w, rules=[(w.target_params, w.draft_params)] * 64, eos_token=eos)
    c = compare_sample(ex, ref, w)
    assert c["n"] == 64 and c["flagged"] + c["boundary"] <= 3, c
    nem = ex.num_emitted.cpu().numpy()
    for b, r in enumerate(ref.seqs):
        if r.accept_margin >= 1e-6 and not r.draft_ambiguous:
            assert nem[b] == r.num_emitted, (b, nem[b], r.num_emitted)
    st = ex.status.cpu().numpy()
    for b, r in enumerate(ref.seqs):                 # the EOS flag where the oracle's block ends in it
        if r.accept_margin >= 1e-6 and not r.draft_ambiguous and not r.status & oracle.SEQ_ERROR_MASK:
            assert bool(st[b] & oracle.SEQ_FLAG_EOS) == bool(r.status & oracle.SEQ_FLAG_EOS), b


def test_greedy_trees_full_batch_sampled():
    """Draft trees over the greedy-at-scale rows (B=256, 9 nodes, V=152064 bf16), the
    benchmark's tree recipe: 64 sequences recomputed by the oracle, bit-exact."""
    import oracle
    import speculative_decoding_verification_44_gb300 as sv
    w = make(4)
    B, N, V = w.B, w.G + 1, w.V
    rng = np.random.default_rng(5000)
    arg = w.target_logits.float().argmax(dim=-1).cpu().numpy()
    tok = np.zeros((B, N), dtype=np.int32)
    par = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        for i in range(1, N):
            par[b, i] = rng.integers(0, i)
            tok[b, i] = arg[b, par[b, i]] if rng.random() < 0.8 else rng.integers(0, V)
    out, path = sv.verify_greedy_tree(w.target_logits, torch.from_numpy(tok).cuda(), torch.from_numpy(par).cuda())
    torch.cuda.synchronize()
    seqs = list(range(0, 256, 4))
    tl = w.target_logits[seqs].float().double().cpu().numpy()
    ref = oracle.verify_greedy_tree(tl, tok[seqs], par[seqs])
    np.testing.assert_array_equal(out.tokens.cpu().numpy()[seqs], ref.tokens)
    np.testing.assert_array_equal(out.num_accepted.cpu().numpy()[seqs], ref.num_accepted)
    P = path.cpu().numpy()[seqs]
    for k, r in enumerate(ref.seqs):
        assert list(P[k, : r.num_accepted + 1]) == r.path


def test_ragged_full_batch_early_exit():
    """The ragged workload at full size (B=512, V=256000) with early exit, as the
    benchmark's --early-exit runs it: the same outputs as the all-rows call (a_i up
    to each stop), and the oracle's early-exit reading on sampled sequences."""
    w = make(5)
    full = gpu_sample(w)
    early = gpu_sample(w, early_exit=True)
    torch.cuda.synchronize()
    for n in ("tokens", "num_accepted", "status", "residual_z"):
        assert torch.equal(getattr(early, n), getattr(full, n)), n
    j = full.num_accepted.cpu().numpy()
    ae, af = early.accept_prob.cpu().numpy(), full.accept_prob.cpu().numpy()
    for b in range(w.B):
        np.testing.assert_array_equal(ae[b, : j[b] + 1], af[b, : j[b] + 1])
        assert (ae[b, j[b] + 1:] == -1).all(), b
    seqs = list(range(3, 512, 16))
    c = compare_sample(early, run_oracle_sample(w, seqs, early_exit=True), w, seqs, early=True)
    assert c["n"] == len(seqs) and c["flagged"] + c["boundary"] <= 3, c
