"""GPU edge cases: data errors reported per sequence, degenerate shapes,
unaligned layouts, workspace reuse.  Every failure is made on the host (bad
values in the inputs); nothing here can fault or hang the GPU."""
import numpy as np
import pytest
import torch

import oracle
from helpers import compare_sample, gpu_greedy, gpu_sample, oracle_probs, run_oracle_greedy, run_oracle_sample, compare_greedy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_verification_44_gb300 import build
    build.build()


def workload(wid, **kw):
    from speculative_decoding_verification_44_gb300 import workloads
    return workloads.make(wid, "cpu", draft_probs=oracle_probs, **kw)


def test_data_errors_commit_nothing():
    w = workload(3, B=10, V=2048)
    w.gamma_per_seq = torch.full((10,), 5, dtype=torch.int32)
    w.gamma_per_seq[0] = 6                         # bad length
    w.gamma_per_seq[1] = -1                        # bad length
    w.draft_tokens[2, 1] = 2048                    # bad token
    w.draft_tokens[3, 4] = -5                      # bad token
    w.u_accept[4, 0] = 1.0                         # bad uniform
    w.u_sample[5] = float("nan")                   # bad uniform
    w.target_logits[6, 2, 17] = float("nan")       # non-finite
    w.draft_logits[7, 0, 5] = float("inf")         # non-finite
    w.target_logits[8, 5] = -float("inf")          # empty support (bonus row)
    w.gamma_per_seq[9] = 2
    w.target_logits[9, 4, 0] = float("nan")        # row beyond gamma_b: never read
    wc = w.to("cuda")
    out = gpu_sample(wc)
    ref = run_oracle_sample(w)
    st = out.status.cpu().tolist()
    assert [s & 0xFF for s in st[:9]] == [1, 1, 2, 2, 3, 3, 4, 4, 5]
    assert st[9] & 0xFF == 0
    compare_sample(out, ref, w)


def test_greedy_data_errors():
    w = workload(4, B=5, V=1000)
    w.gamma_per_seq = torch.tensor([8, 9, 3, 8, 2], dtype=torch.int32)
    w.draft_tokens[2, 0] = 1000
    w.target_logits[3, 8, 3] = float("nan")
    w.target_logits[4, 1] = -float("inf")
    out = gpu_greedy(w.to("cuda"))
    assert [s & 0xFF for s in out.status.cpu().tolist()] == [0, 1, 2, 4, 5]
    compare_greedy(out, run_oracle_greedy(w), w)


@pytest.mark.parametrize("V", [1, 2, 7, 33, 1000003 // 97])
def test_small_and_odd_vocabularies(V):
    w = workload(1, B=64, V=V)
    c = compare_sample(gpu_sample(w.to("cuda")), run_oracle_sample(w), w)
    assert c["n"] == 64


def test_unaligned_base_pointer_uses_element_path():
    """A logits tensor that starts 2 bytes past a 16-byte boundary."""
    w = workload(3, B=6, V=4096)
    wc = w.to("cuda")
    big = torch.empty(wc.target_logits.numel() + 8, dtype=torch.bfloat16, device="cuda")
    view = big[1:1 + wc.target_logits.numel()].view_as(wc.target_logits)
    view.copy_(wc.target_logits)
    assert view.data_ptr() % 16 == 2
    wc.target_logits = view
    compare_sample(gpu_sample(wc), run_oracle_sample(w), w)


def test_workspace_reuse_and_counters_reset():
    import speculative_decoding_verification_44_gb300 as sv
    w = workload(3, B=16, V=4096)
    wc = w.to("cuda")
    ws = sv.new_workspace(sv.workspace_size(w.B, w.G, w.V, w.target_params, w.draft_params), "cuda")
    o1 = gpu_sample(wc, workspace=ws)
    torch.cuda.synchronize()
    assert (ws[: 4 * w.B] == 0).all()               # counter region restored to zero
    o2 = gpu_sample(wc, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1.tokens, o2.tokens) and torch.equal(o1.num_accepted, o2.num_accepted)
    # full-row target rows: the draw runs chunk-parallel in a second kernel with
    # its own per-sequence counters, right after the row counters
    f = workload(5, B=8, V=9000)
    fc = f.to("cuda")
    fws = sv.new_workspace(sv.workspace_size(f.B, f.G, f.V, f.target_params, f.draft_params), "cuda")
    zero = 2 * ((4 * f.B + 255) // 256 * 256)
    f1 = gpu_sample(fc, workspace=fws)
    torch.cuda.synchronize()
    assert (fws[:zero] == 0).all()
    f2 = gpu_sample(fc, workspace=fws)
    torch.cuda.synchronize()
    assert torch.equal(f1.tokens, f2.tokens) and torch.equal(f1.status, f2.status)
    assert torch.equal(f1.residual_z, f2.residual_z)
    g = workload(4, B=8, V=4096).to("cuda")
    gws = sv.new_workspace(sv.greedy_workspace_size(g.B, g.G), "cuda")
    for _ in range(3):
        gpu_greedy(g, workspace=gws)
    torch.cuda.synchronize()
    assert (gws[: 4 * g.B] == 0).all()


def test_draft_token_with_zero_draft_probability_is_flagged():
    """q(d) = 0 (a draft token outside the draft's own top-k)."""
    w = workload(3, B=4, V=4096)
    for b in range(4):
        row = w.draft_logits[b, 0].float()
        w.draft_tokens[b, 0] = int(row.argmin())
    wc = w.to("cuda")
    out = gpu_sample(wc)
    ref = run_oracle_sample(w)
    assert all(s.status & oracle.SEQ_FLAG_ZERO_Q for s in ref.seqs)
    assert (out.status.cpu() & 0x100).all()
    compare_sample(out, ref, w)


def test_identical_target_and_draft_accept_everything():
    w = workload(3, B=8, V=4096)
    w.draft_logits = w.target_logits[:, : w.G].clone()
    from speculative_decoding_verification_44_gb300.workloads import sample_from_probs
    q = oracle_probs(w.draft_logits.reshape(-1, w.V), w.draft_params)
    w.draft_tokens = sample_from_probs(q, torch.Generator().manual_seed(1)).reshape(w.B, w.G).to(torch.int32)
    out = gpu_sample(w.to("cuda"))
    assert (out.num_accepted.cpu() == w.G).all()
    assert (out.accept_prob.cpu() == 1.0).all()
