"""Top-p cuts whose crossing value is shared by many tokens.

A full-row top-p row on the value-count path leaves open which of the cut
value's ties come first (R2: the first n in index order are kept): the row
records only n, the draft token's probability is decided by the token's rank
among the ties, and the full-row draw corrects its chunk sums by tie counts
and re-scans the one chunk where the n-th tie falls.  These rows take their
logits from a few levels, so every cut value has hundreds of ties and the cut
falls inside a tie class; draft tokens are chosen among the ties of the target's
cut value on both sides of the n-th one.  Results must match the float64 oracle
under the usual boundary rules [wrblog §7.3; R2, R3]."""
import numpy as np
import pytest
import torch

import oracle
from helpers import compare_sample, gpu_sample, run_oracle_sample

pytestmark = pytest.mark.gpu

LEVELS = np.array([3.0, 2.0, 1.5, 1.0, 0.5, -1.0])   # exact in bf16
WEIGHTS = [0.002, 0.01, 0.05, 0.2, 0.4, 0.338]


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_verification_44_gb300 import build
    build.build()


def make(seed, B=24, G=3, V=40960, top_p=0.537):
    """Leveled rows (target and draft), draft tokens among the target cut's ties."""
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300.workloads import Workload
    rng = np.random.default_rng(seed)
    zt = LEVELS[rng.choice(len(LEVELS), size=(B, G + 1, V), p=WEIGHTS)].astype(np.float32)
    zd = LEVELS[rng.choice(len(LEVELS), size=(B, G, V), p=WEIGHTS)].astype(np.float32)
    toks = np.zeros((B, G), dtype=np.int32)
    partial = on_kept = on_dropped = 0
    for b in range(B):
        for i in range(G):
            row = zt[b, i].astype(np.float64)
            kept = oracle.transform_row(row, 1.0, 0, top_p).kept
            cut = row[kept[-1]]
            ties = np.flatnonzero(row == cut)                 # index order
            n = int(np.sum(row[kept] == cut))                 # ties the prefix keeps
            partial += int(0 < n < len(ties))
            pick = (b + i) % 3
            if pick == 0 and n > 0:
                toks[b, i] = ties[rng.integers(0, n)]
                on_kept += 1
            elif pick == 1 and n < len(ties):
                toks[b, i] = ties[rng.integers(n, len(ties))]
                on_dropped += 1
            else:
                toks[b, i] = rng.integers(0, V)
    params = sv.SamplingParams(1.0, 0, top_p)
    w = Workload("leveled-ties", 0, "sample", B, G, V, torch.bfloat16, params, params)
    dev = torch.device("cuda")
    w.target_logits = torch.from_numpy(zt).to(torch.bfloat16).to(dev)
    w.draft_logits = torch.from_numpy(zd).to(torch.bfloat16).to(dev)
    w.draft_tokens = torch.from_numpy(toks).to(dev)
    w.draft_is_onehot = (torch.arange(B, device=dev) % 2).to(torch.uint8)   # both draw modes
    g = torch.Generator(device="cpu").manual_seed(seed)
    w.u_accept = torch.rand(B, G, generator=g).to(dev)
    w.u_sample = torch.rand(B, generator=g).to(dev)
    return w, partial, on_kept, on_dropped


@pytest.mark.parametrize("seed,top_p", [(5, 0.537), (6, 0.711), (7, 0.912)])
def test_leveled_rows_match_oracle(seed, top_p):
    w, partial, on_kept, on_dropped = make(seed, top_p=top_p)
    # the cases this test exists for: cuts inside a tie class, draft tokens on both sides
    assert partial >= w.B * w.G // 2 and on_kept >= 5 and on_dropped >= 5, (partial, on_kept, on_dropped)
    out = gpu_sample(w)
    torch.cuda.synchronize()
    ref = run_oracle_sample(w)
    c = compare_sample(out, ref, w)
    assert c["flagged"] + c["boundary"] <= max(2, 0.02 * c["n"]), c
    assert c["exact"] >= 0.9 * (c["n"] - c["flagged"] - c["errors"]), c
    assert c["rejected"] > 0, c


def test_dropped_ties_have_zero_probability():
    """A draft token among the cut value's ties but past the n-th has p = 0 and is rejected."""
    w, _, _, on_dropped = make(8)
    assert on_dropped > 0
    out = gpu_sample(w)
    torch.cuda.synchronize()
    ref = run_oracle_sample(w)
    aprob = out.accept_prob.cpu().numpy()
    for k in range(w.B):
        r = ref.seqs[k]
        for i in range(min(int(r.num_accepted) + 1, w.G)):
            if r.accept_prob[i] == 0.0:
                assert aprob[k, i] == 0.0, (k, i, aprob[k, i])
