"""The allocation-free sampling entry point, spec_verify_sample_noalloc.

Some callers cannot hand the library a workspace: a plugin inside an
inference server whose device memory is owned by the server's allocator, or a
latency-critical path that must not pay cudaMalloc's device-wide
synchronisation.  For them the library keeps its scratch in a fixed 8 MiB
array of its own device memory.  This test calls that entry point through the
C ABI twice in a row and checks both results against spec_verify_sample on the
same inputs (every output bit for bit: the same kernels run on the same
inputs), that a request needing more than 8 MiB of scratch is refused before
launching, and that a call refused by the host checks writes nothing and does
not disturb the calls around it.

It sits in its own file, collected last, so a stop-at-first-failure run has
already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from speculative_decoding_verification_44_gb300 import build, _lib
    build.build()
    return _lib


def serving_inputs(B, V, seed):
    """Zipf-shaped bf16 logits (the serving recipe) with arbitrary draft tokens."""
    from speculative_decoding_verification_44_gb300 import workloads, SamplingParams
    g = torch.Generator(device="cuda").manual_seed(seed)
    G = 5
    tgt = workloads._zipf_rows(B * (G + 1), V, g, 0.5, "cuda").view(B, G + 1, V)
    dft = (tgt[:, :G] + 0.8 * torch.randn(B, G, V, generator=g, device="cuda")).to(torch.bfloat16)
    tgt = tgt.to(torch.bfloat16).contiguous()
    # draft tokens: mostly the draft row's argmax (likely kept by top-k), some random
    toks = dft.float().argmax(dim=2)
    rnd = torch.randint(0, V, (B, G), generator=g, device="cuda")
    toks = torch.where(torch.rand(B, G, generator=g, device="cuda") < 0.8, toks, rnd).to(torch.int32)
    ua = torch.rand(B, G, generator=g, device="cuda")
    us = torch.rand(B, generator=g, device="cuda")
    p = SamplingParams(0.7, 50, 0.9)
    return dict(tgt=tgt, dft=dft.contiguous(), toks=toks.contiguous(), ua=ua, us=us, p=p, B=B, G=G, V=V)


def outputs(B, G):
    return dict(tokens=torch.full((B, G + 1), -7, dtype=torch.int32, device="cuda"),
                nacc=torch.full((B,), -7, dtype=torch.int32, device="cuda"),
                aprob=torch.full((B, G), -7.0, dtype=torch.float32, device="cuda"),
                z=torch.full((B,), -7.0, dtype=torch.float32, device="cuda"),
                status=torch.full((B,), -7, dtype=torch.int32, device="cuda"))


def call_noalloc(lib, x, o):
    s = torch.cuda.current_stream().cuda_stream
    return lib.spec_verify_sample_noalloc(
        x["tgt"].data_ptr(), x["dft"].data_ptr(), lib.SPEC_BF16, x["toks"].data_ptr(), None, None,
        x["ua"].data_ptr(), x["us"].data_ptr(), x["p"].c(), x["p"].c(), x["B"], x["G"], x["V"],
        o["tokens"].data_ptr(), o["nacc"].data_ptr(), o["aprob"].data_ptr(), o["z"].data_ptr(),
        o["status"].data_ptr(), s)


def call_with_workspace(lib, x, o):
    from speculative_decoding_verification_44_gb300 import new_workspace, workspace_size
    ws = new_workspace(workspace_size(x["B"], x["G"], x["V"], x["p"], x["p"]), "cuda")
    s = torch.cuda.current_stream().cuda_stream
    return lib.spec_verify_sample(
        x["tgt"].data_ptr(), x["dft"].data_ptr(), lib.SPEC_BF16, x["toks"].data_ptr(), None, None,
        x["ua"].data_ptr(), x["us"].data_ptr(), x["p"].c(), x["p"].c(), x["B"], x["G"], x["V"],
        ws.data_ptr(), ws.numel(), o["tokens"].data_ptr(), o["nacc"].data_ptr(), o["aprob"].data_ptr(),
        o["z"].data_ptr(), o["status"].data_ptr(), s), ws


@pytest.mark.parametrize("B", [16, 64])
def test_noalloc_matches_workspace_entry_point_on_two_calls(lib, B):
    x = serving_inputs(B, 128256, seed=B)
    ref = outputs(B, x["G"])
    st, ws = call_with_workspace(lib, x, ref)
    assert st == lib.SPEC_OK
    torch.cuda.synchronize()
    for _ in range(2):                       # two calls in a row share the static scratch
        got = outputs(B, x["G"])
        assert call_noalloc(lib, x, got) == lib.SPEC_OK
        torch.cuda.synchronize()
        assert torch.equal(got["tokens"], ref["tokens"])
        assert torch.equal(got["nacc"], ref["nacc"])
        assert torch.equal(got["status"], ref["status"])
        # the same kernels on the same inputs: the probabilities agree bit for bit
        assert torch.equal(got["aprob"], ref["aprob"])
        assert torch.equal(got["z"], ref["z"])
    assert (ref["nacc"].cpu() >= 0).all()


def test_noalloc_refuses_requests_beyond_its_scratch(lib):
    x = serving_inputs(2, 4096, seed=3)
    o = outputs(2, x["G"])
    big_batch = 4096                          # needs about 94 MB of workspace with top-k 50
    s = torch.cuda.current_stream().cuda_stream
    st = lib.spec_verify_sample_noalloc(
        x["tgt"].data_ptr(), x["dft"].data_ptr(), lib.SPEC_BF16, x["toks"].data_ptr(), None, None,
        x["ua"].data_ptr(), x["us"].data_ptr(), x["p"].c(), x["p"].c(), big_batch, x["G"], x["V"],
        o["tokens"].data_ptr(), o["nacc"].data_ptr(), o["aprob"].data_ptr(), o["z"].data_ptr(),
        o["status"].data_ptr(), s)
    assert st == lib.SPEC_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (o["tokens"].cpu() == -7).all()   # nothing was launched


def test_noalloc_invalid_call_launches_nothing(lib):
    """A call refused by the host checks (here a misaligned output pointer)
    returns its status with nothing written, and the valid calls before and
    after it still match the workspace entry point."""
    x = serving_inputs(8, 128256, seed=11)
    ref = outputs(8, x["G"])
    st, ws = call_with_workspace(lib, x, ref)
    assert st == lib.SPEC_OK
    got = outputs(8, x["G"])
    assert call_noalloc(lib, x, got) == lib.SPEC_OK
    bad = outputs(8, x["G"])
    s = torch.cuda.current_stream().cuda_stream
    st = lib.spec_verify_sample_noalloc(
        x["tgt"].data_ptr(), x["dft"].data_ptr(), lib.SPEC_BF16, x["toks"].data_ptr(), None, None,
        x["ua"].data_ptr(), x["us"].data_ptr(), x["p"].c(), x["p"].c(), x["B"], x["G"], x["V"],
        bad["tokens"].data_ptr() + 2, bad["nacc"].data_ptr(), bad["aprob"].data_ptr(), bad["z"].data_ptr(),
        bad["status"].data_ptr(), s)
    assert st == lib.SPEC_ERR_MISALIGNED
    torch.cuda.synchronize()
    assert (bad["tokens"].cpu() == -7).all()
    for k in ref:
        assert torch.equal(got[k], ref[k]), k
    again = outputs(8, x["G"])
    assert call_noalloc(lib, x, again) == lib.SPEC_OK
    torch.cuda.synchronize()
    for k in ref:
        assert torch.equal(again[k], ref[k]), k
