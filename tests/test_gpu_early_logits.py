"""Early logits reads (spec_set_early_logits_reads): the kept-list, greedy and tree
verifiers then stream their logits rows before they wait for the previous call in the
stream, so back-to-back calls overlap on the GPU.  Calls issued back to back with the
switch on must give exactly the results of the same calls with it off (each call waits
for the previous one before it reads anything else or writes anything), including when
consecutive calls share one workspace."""
import numpy as np
import pytest
import torch

from test_gpu_tree import make_trees
from test_gpu_tree_sample import make_sample_trees

pytestmark = pytest.mark.gpu

ROUNDS = 3


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_verification_44_gb300 import build
    build.build()
    import speculative_decoding_verification_44_gb300 as sv
    yield
    sv.set_early_logits_reads(False)


def _both(run):
    """run() issues calls back to back and returns their outputs; compare off vs on."""
    import speculative_decoding_verification_44_gb300 as sv
    try:
        sv.set_early_logits_reads(False)
        a = run()
        torch.cuda.synchronize()
        sv.set_early_logits_reads(True)
        b = run()
        torch.cuda.synchronize()
    finally:
        sv.set_early_logits_reads(False)
    assert len(a) == len(b)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    return a


def _outs(o, names=("tokens", "num_accepted", "status", "accept_prob", "residual_z")):
    return [getattr(o, n).clone() for n in names if getattr(o, n) is not None]


def test_serving_calls_back_to_back():
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import workloads
    dev = torch.device("cuda")
    dp = lambda rows, params: sv.transform_probs(rows.contiguous(), params)[0]   # noqa: E731
    sets = [workloads.make(3, dev, B=16, draft_probs=dp, replica=r) for r in range(4)]
    w0 = sets[0]
    ws = sv.new_workspace(sv.workspace_size(w0.B, w0.G, w0.V, w0.target_params, w0.draft_params), dev)

    def run():
        res = []
        for _ in range(ROUNDS):
            outs = [sv.alloc_outputs(w0.B, w0.G, dev) for _ in sets]
            for w, o in zip(sets, outs):
                sv.verify_sample(w.target_logits, w.draft_logits, w.draft_tokens, w.u_accept, w.u_sample,
                                 w.target_params, w.draft_params, workspace=ws, out=o)
            for o in outs:
                res += _outs(o)
        return res

    res = _both(run)
    assert all((t == 0).all() for t in res[2::5])          # status: every sequence valid


def test_greedy_calls_back_to_back():
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import workloads
    dev = torch.device("cuda")
    sets = [workloads.make(4, dev, B=16, replica=r) for r in range(4)]
    w0 = sets[0]
    ws = sv.new_workspace(sv.greedy_workspace_size(w0.B, w0.G), dev)

    def run():
        res = []
        for _ in range(ROUNDS):
            outs = [sv.verify_greedy(w.target_logits, w.draft_tokens, workspace=ws) for w in sets]
            for o in outs:
                res += _outs(o, ("tokens", "num_accepted", "status"))
        return res

    _both(run)


def test_tree_calls_back_to_back():
    import speculative_decoding_verification_44_gb300 as sv
    logits, tokens, parents = make_trees(8, 9, 4096, torch.bfloat16, seed=71)
    logits, tokens, parents = logits.cuda(), tokens.cuda(), parents.cuda()
    tp = sv.SamplingParams(0.7, 50, 0.9)
    tgt, dft, stok, spar, u_node, u_sample = make_sample_trees(8, 6, 4096, torch.bfloat16, 72, tp, tp)
    tgt, dft, stok, spar = tgt.cuda(), dft.cuda(), stok.cuda(), spar.cuda()
    u_node, u_sample = u_node.cuda(), u_sample.cuda()

    def run():
        res = []
        for _ in range(ROUNDS):
            for _ in range(2):
                out, path = sv.verify_greedy_tree(logits, tokens, parents)
                res += _outs(out, ("tokens", "num_accepted", "status")) + [path.clone()]
                out, path = sv.verify_sample_tree(tgt, dft, stok, spar, u_node, u_sample, tp, tp)
                res += _outs(out) + [path.clone()]
        return res

    _both(run)


def test_switch_defaults_off_and_is_a_plain_setting():
    import speculative_decoding_verification_44_gb300 as sv
    from speculative_decoding_verification_44_gb300 import _lib
    lib = _lib.load()
    assert lib.spec_set_early_logits_reads(1) == 0
    assert lib.spec_set_early_logits_reads(0) == 0
    sv.set_early_logits_reads(False)
    assert np.isscalar(_lib.SPEC_SEQ_STALLED)
