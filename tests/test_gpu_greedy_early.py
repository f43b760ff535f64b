"""GPU parity of early-exit greedy verification (spec_verify_greedy_early).

The CUDA path skips a sequence's rows once an earlier row has failed or
mismatched, and forms the result from the rows up to that stop; the oracle's
verify_greedy_early reads rows in order and stops there (reading R11).
Tokens, accepted counts and statuses must agree exactly.  Rows whose
predecessors were still running when they were scheduled are read
speculatively, so the rows read lie between the oracle's count and
gamma_b + 1.  On valid inputs the result also equals the all-rows verifier.
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


def workload(**kw):
    from speculative_decoding_verification_44_gb300 import workloads
    return workloads.make(4, "cpu", **kw).to("cuda")


def run_early(w):
    import speculative_decoding_verification_44_gb300 as sv
    rows = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    out = sv.verify_greedy_early(w.target_logits, w.draft_tokens, w.gamma_per_seq, rows_read=rows)
    torch.cuda.synchronize()
    return out, rows.cpu().numpy()


def oracle_early(w, seqs=None):
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    gam = None if w.gamma_per_seq is None else w.gamma_per_seq.cpu().numpy()[seqs]
    return oracle.verify_greedy_early(to_f64(w.target_logits[seqs]), w.draft_tokens.cpu().numpy()[seqs], gam)


def compare(out, rows, ref, seqs, gammas):
    toks, nacc, status = out.tokens.cpu().numpy(), out.num_accepted.cpu().numpy(), out.status.cpu().numpy()
    for k, b in enumerate(seqs):
        r = ref.seqs[k]
        assert status[b] == r.status, (b, status[b], r.status)
        assert nacc[b] == r.num_accepted, (b, nacc[b], r.num_accepted)
        assert (toks[b] == r.tokens).all(), (b, toks[b], r.tokens)
        if r.rows_read < 0:
            assert rows[b] == 0, (b, rows[b])
        else:
            assert r.rows_read <= rows[b] <= gammas[b] + 1, (b, rows[b], r.rows_read)


def gammas_of(w):
    return (w.gamma_per_seq.cpu().numpy() if w.gamma_per_seq is not None
            else np.full(w.B, w.G))


@pytest.mark.parametrize("V", [4096, 5003, 32000])
def test_matches_oracle(V):
    w = workload(B=40, V=V)
    out, rows = run_early(w)
    compare(out, rows, oracle_early(w), range(w.B), gammas_of(w))


def test_ragged_gammas_and_zero():
    w = workload(B=24, V=4096)
    w.gamma_per_seq = torch.tensor([i % (w.G + 1) for i in range(w.B)], dtype=torch.int32, device="cuda")
    out, rows = run_early(w)
    compare(out, rows, oracle_early(w), range(w.B), gammas_of(w))
    assert (rows[w.gamma_per_seq.cpu().numpy() == 0] == 1).all()


def test_full_size_equals_all_rows_greedy_and_oracle_sample():
    """Greedy at scale (B=256, gamma=8, V=152064 bf16): identical to the all-rows
    verifier everywhere; oracle-exact on a sample of sequences."""
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import workloads
    w = workloads.make(4, "cuda")
    out, rows = run_early(w)
    full = sv.verify_greedy(w.target_logits, w.draft_tokens, w.gamma_per_seq)
    torch.cuda.synchronize()
    assert torch.equal(out.tokens, full.tokens)
    assert torch.equal(out.num_accepted, full.num_accepted)
    assert torch.equal(out.status, full.status)
    nacc = out.num_accepted.cpu().numpy()
    assert ((rows >= nacc + 1) & (rows <= w.G + 1)).all()
    # 2304 row CTAs run in several waves: rows of decided sequences are skipped
    assert rows.mean() < w.G + 1 - 1.0, rows.mean()
    seqs = list(range(0, w.B, 16))
    compare(out, rows, oracle_early(w, seqs), seqs, gammas_of(w))


def test_rows_after_the_stop_do_not_affect_the_result():
    """A NaN row after the first mismatch does not fail the sequence; at or
    before the stop it does.  Length and token errors come first."""
    import speculative_decoding_verification_44_gb300 as sv
    B, G, V = 6, 4, 3000
    z = torch.zeros(B, G + 1, V)
    z[:, :, 5] = 2.0                                     # argmax 5 on every row
    toks = torch.full((B, G), 5, dtype=torch.int32)
    toks[:, 2] = 9                                       # first mismatch at position 2
    z[0, 3, 17] = float("nan")                           # after the stop: ignored
    z[1, 4, :] = float("nan")                            # bonus row after the stop: ignored
    z[2, 2, 17] = float("nan")                           # at the stop: NONFINITE
    z[3, 1, :] = -float("inf")                           # before the stop: EMPTY_SUPPORT
    toks[4, 0] = V                                       # bad token, even with clean rows
    gam = torch.full((B,), G, dtype=torch.int32)
    gam[5] = G + 1                                       # bad length
    zc = z.to(torch.bfloat16).cuda()
    rows = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out = sv.verify_greedy_early(zc, toks.cuda(), gam.cuda(), rows_read=rows)
    torch.cuda.synchronize()
    st = out.status.cpu().tolist()
    assert st == [oracle.SEQ_OK, oracle.SEQ_OK, oracle.SEQ_NONFINITE, oracle.SEQ_EMPTY_SUPPORT,
                  oracle.SEQ_BAD_TOKEN, oracle.SEQ_BAD_LENGTH]
    assert out.num_accepted.cpu().tolist() == [2, 2, -1, -1, -1, -1]
    assert out.tokens[0].cpu().tolist() == [5, 5, 5, -1, -1]
    ref = oracle.verify_greedy_early(to_f64(zc), toks.numpy(), gam.numpy())
    assert [r.status for r in ref.seqs] == st
    rr = rows.cpu().tolist()
    assert rr[4:] == [0, 0]
    assert all(r.rows_read <= rr[b] <= G + 1 for b, r in enumerate(ref.seqs[:4]))
    # the all-rows verifier fails the first two sequences on rows it must read
    full = sv.verify_greedy(zc, toks.cuda(), gam.cuda())
    torch.cuda.synchronize()
    assert full.status.cpu().tolist()[:2] == [oracle.SEQ_NONFINITE, oracle.SEQ_NONFINITE]


def test_ties_pick_lowest_index_and_float32():
    import speculative_decoding_verification_44_gb300 as sv
    V = 3001
    z = torch.zeros(1, 3, V, dtype=torch.float32)
    z[0, 0, [50, 7, 3000]] = 4.0        # argmax 7
    z[0, 1, [1, 0]] = 3.0               # argmax 0
    z[0, 2, 100] = -0.0                 # all zero: argmax 0 (-0 == +0)
    toks = torch.tensor([[7, 0]], dtype=torch.int32)
    rows = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = sv.verify_greedy_early(z.cuda(), toks.cuda(), rows_read=rows)
    torch.cuda.synchronize()
    assert out.num_accepted.item() == 2 and rows.item() == 3            # every row was needed
    assert out.tokens.cpu().tolist() == [[7, 0, 0]]
