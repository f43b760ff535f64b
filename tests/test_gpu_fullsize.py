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
