"""Shared test utilities: oracle-backed draft sampling and GPU-vs-oracle comparison.

Boundary rules (the tolerance the parity tests state):
* accept counts and greedy tokens are bit-exact, except sequences where some
  evaluated |u_i - a_i| < 1e-6, or an evaluated draft token or the drawn token
  is one whose top-p membership turns on a cumulative probability within 1e-6
  of top_p ("flagged": counted, outputs checked for validity only);
* a sampled token may differ from the oracle's only when u lies within 1e-6
  of every normalised CDF boundary between the two tokens ("boundary");
* probabilities (a_i, Z, transformed rows) agree within 1e-5 absolute.
"""
import numpy as np
import torch

import oracle

TOL_PROB = 1e-5
TOL_BOUNDARY = 1e-6


def f32(x):
    """The float32 value a parameter has inside the library, as a Python float."""
    return float(np.float32(x))


def params_tuple(p):
    return (f32(p.temperature), int(p.top_k), f32(p.top_p))


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").float().double().numpy()


def oracle_probs(rows: torch.Tensor, params) -> torch.Tensor:
    """Draft distribution q from the float64 oracle (used to draw draft tokens)."""
    p, _ = oracle.transform_rows(to_f64(rows), *params_tuple(params))
    return torch.from_numpy(p)


def run_oracle_sample(w, seqs=None, keep_cdf=True, lenience=1.0, rules=None, eos_token=-1, early_exit=False):
    """The oracle on workload ``w``; ``rules``: per sequence (target SamplingParams, draft SamplingParams)."""
    tl = to_f64(w.target_logits) if seqs is None else to_f64(w.target_logits[seqs])
    dl = None
    if w.draft_logits is not None:
        dl = to_f64(w.draft_logits) if seqs is None else to_f64(w.draft_logits[seqs])
    sel = slice(None) if seqs is None else seqs
    toks = w.draft_tokens.cpu().numpy()[sel]
    ua = w.u_accept.cpu().double().numpy()[sel]
    us = w.u_sample.cpu().double().numpy()[sel]
    gam = None if w.gamma_per_seq is None else w.gamma_per_seq.cpu().numpy()[sel]
    oh = None if w.draft_is_onehot is None else w.draft_is_onehot.cpu().numpy()[sel]
    per = None
    if rules is not None:
        per = [(params_tuple(t), params_tuple(d)) for t, d in rules]
        if seqs is not None:
            per = [per[b] for b in seqs]
    return oracle.verify_sample(tl, dl, toks, ua, us, params_tuple(w.target_params),
                                params_tuple(w.draft_params), gam, oh, keep_cdf=keep_cdf,
                                lenience=lenience, params_per_seq=per, eos_token=eos_token,
                                early_exit=early_exit)


def run_oracle_greedy(w, seqs=None):
    sel = slice(None) if seqs is None else seqs
    tl = to_f64(w.target_logits) if seqs is None else to_f64(w.target_logits[seqs])
    gam = None if w.gamma_per_seq is None else w.gamma_per_seq.cpu().numpy()[sel]
    return oracle.verify_greedy(tl, w.draft_tokens.cpu().numpy()[sel], gam)


def gpu_sample(w, **kw):
    import speculative_decoding_verification_44_gb300 as sv
    return sv.verify_sample(w.target_logits, w.draft_logits, w.draft_tokens, w.u_accept, w.u_sample,
                            w.target_params, w.draft_params, w.gamma_per_seq, w.draft_is_onehot, **kw)


def gpu_greedy(w, **kw):
    import speculative_decoding_verification_44_gb300 as sv
    return sv.verify_greedy(w.target_logits, w.draft_tokens, w.gamma_per_seq, **kw)


def compare_sample(out, ref, w, seqs=None, early=False):
    """Element-by-element comparison under the boundary rules; returns counters.
    ``early``: early-exit results, whose a_i stop at each side's own stop."""
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    toks = out.tokens.cpu().numpy()
    nacc = out.num_accepted.cpu().numpy()
    status = out.status.cpu().numpy()
    aprob = out.accept_prob.cpu().numpy() if out.accept_prob is not None else None
    zres = out.residual_z.cpu().numpy() if out.residual_z is not None else None
    gam_all = (w.gamma_per_seq.cpu().numpy() if w.gamma_per_seq is not None
               else np.full(w.B, w.G))
    us = w.u_sample.cpu().double().numpy()
    c = dict(n=0, exact=0, flagged=0, boundary=0, errors=0, rejected=0, bonus=0)
    for k, b in enumerate(seqs):
        r = ref.seqs[k]
        c["n"] += 1
        gb = int(gam_all[b])
        if r.status & oracle.SEQ_ERROR_MASK:
            assert (status[b] & 0xFF) == (r.status & 0xFF), (b, status[b], r.status)
            assert nacc[b] == -1 and (toks[b] == -1).all(), b
            c["errors"] += 1
            continue
        assert (status[b] & 0xFF) == 0, (b, status[b])
        n = int(nacc[b])
        assert 0 <= n <= gb, (b, n, gb)
        if r.num_emitted == r.num_accepted:         # the oracle's block ends at an accepted EOS draft
            if r.accept_margin < TOL_BOUNDARY or r.draft_ambiguous:
                c["flagged"] += 1
                continue
            assert n == r.num_accepted and (toks[b] == r.tokens).all(), (b, toks[b], r.tokens)
            assert status[b] & oracle.SEQ_FLAG_EOS, (b, status[b])
            c["eos_cut"] = c.get("eos_cut", 0) + 1
            c["exact"] += 1
            continue
        assert 0 <= toks[b, n] < w.V, (b, toks[b])
        assert (toks[b, n + 1:] == -1).all(), (b, toks[b])
        if aprob is not None and early:
            k = min(n, r.num_accepted, gb - 1) + 1           # positions both sides decided
            np.testing.assert_allclose(aprob[b, :k], r.accept_prob[:k], atol=TOL_PROB, rtol=0,
                                       err_msg=f"accept_prob seq {b}")
            assert (aprob[b, n + 1:] == -1).all(), (b, aprob[b])
        elif aprob is not None:
            np.testing.assert_allclose(aprob[b, :gb], r.accept_prob[:gb], atol=TOL_PROB, rtol=0,
                                       err_msg=f"accept_prob seq {b}")
            assert (aprob[b, gb:] == -1).all()
        if (r.accept_margin < TOL_BOUNDARY or r.draft_ambiguous
                or toks[b, n] in r.sample_ambiguous or r.tokens[r.num_accepted] in r.sample_ambiguous):
            c["flagged"] += 1
            continue
        assert n == r.num_accepted, (b, n, r.num_accepted, r.accept_margin)
        assert (toks[b, :n] == r.tokens[:n]).all(), b
        assert (status[b] & 0x100) == (r.status & 0x100), (b, status[b], r.status)
        if n < gb:
            c["rejected"] += 1
            if zres is not None:
                assert abs(zres[b] - r.residual_Z) <= TOL_PROB, (b, zres[b], r.residual_Z)
        else:
            c["bonus"] += 1
            if zres is not None:
                assert zres[b] == -1.0
        g, o = int(toks[b, n]), int(r.tokens[n])
        if g == o:
            c["exact"] += 1
        else:
            cdf = r.sample_cdf
            u = us[b]
            if g < o:
                ok = cdf[g] >= u - TOL_BOUNDARY
            else:
                ok = cdf[g - 1] <= u + TOL_BOUNDARY
            assert ok, (b, g, o, u, cdf[min(g, o)], cdf[max(g, o) - 1])
            c["boundary"] += 1
    return c


def compare_greedy(out, ref, w, seqs=None):
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    toks = out.tokens.cpu().numpy()
    nacc = out.num_accepted.cpu().numpy()
    status = out.status.cpu().numpy()
    for k, b in enumerate(seqs):
        r = ref.seqs[k]
        assert status[b] == r.status, (b, status[b], r.status)
        assert nacc[b] == r.num_accepted, (b, nacc[b], r.num_accepted)
        assert (toks[b] == r.tokens).all(), (b, toks[b], r.tokens)
    return len(seqs)


def check_sample_counts(out, ref, w, seqs=None, min_exact=0.9, early=False):
    """compare_sample plus the parity bar: few flagged / boundary sequences, the rest exact."""
    c = compare_sample(out, ref, w, seqs, early)
    assert c["flagged"] + c["boundary"] <= max(2, 0.02 * c["n"]), c
    assert c["exact"] >= min_exact * (c["n"] - c["flagged"] - c["errors"]), c
    return c
