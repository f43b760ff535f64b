"""Oracle pins for the logits transforms (temperature, top-k, top-p, bf16 widening).

Each check compares the oracle with something other than itself: a library
softmax, a library argmax, or a brute-force set definition.
"""
import itertools

import numpy as np
import pytest
import scipy.special
import torch

import oracle


def test_no_truncation_is_textbook_softmax():
    rng = np.random.default_rng(1)
    for T in (0.3, 0.7, 1.0, 2.5):
        z = rng.normal(0, 3, size=257)
        rd = oracle.transform_row(z, T, 0, 1.0)
        np.testing.assert_allclose(rd.probs, scipy.special.softmax(z / T), rtol=1e-12, atol=1e-15)
        # top_k >= V is also "off"
        np.testing.assert_allclose(oracle.transform_row(z, T, 257, 1.0).probs, rd.probs, atol=0)


def test_top1_is_argmax_one_hot_with_low_index_ties():
    z = np.array([0.5, 2.0, -1.0, 2.0, 1.9])
    rd = oracle.transform_row(z, 0.8, 1, 1.0)
    assert int(np.argmax(z)) == 1                    # library argmax: first maximum
    np.testing.assert_array_equal(rd.probs, np.eye(5)[1])
    # -0.0 and +0.0 tie; the lower index wins
    z = np.array([-0.0, 0.0, -1.0])
    assert oracle.transform_row(z, 1.0, 1, 1.0).probs[0] == 1.0


def test_top_k_matches_counting_definition():
    rng = np.random.default_rng(2)
    for _ in range(50):
        V = int(rng.integers(2, 40))
        z = rng.normal(0, 2, size=V)
        k = int(rng.integers(1, V))
        T = float(rng.uniform(0.2, 2.0))
        rd = oracle.transform_row(z, T, k, 1.0)
        # a token is kept iff fewer than k tokens are strictly larger (distinct logits)
        kept = np.array([(z > z[x]).sum() < k for x in range(V)])
        assert kept.sum() == k
        expect = np.where(kept, np.exp(z / T), 0.0)
        np.testing.assert_allclose(rd.probs, expect / expect.sum(), rtol=1e-12, atol=1e-16)


def test_top_k_ties_keep_lower_indices():
    z = np.array([1.0, 3.0, 1.0, 1.0, 3.0])
    rd = oracle.transform_row(z, 1.0, 3, 1.0)
    assert set(np.flatnonzero(rd.probs)) == {0, 1, 4}


def test_top_p_matches_smallest_set_definition():
    """Nucleus = the smallest token set whose probability reaches top_p (largest mass among
    sets of that size), checked by enumerating every subset for V <= 8."""
    rng = np.random.default_rng(3)
    checked = 0
    for _ in range(300):
        V = int(rng.integers(2, 9))
        z = rng.normal(0, 1.5, size=V)
        T = float(rng.uniform(0.3, 2.0))
        k = int(rng.integers(0, V + 1))
        top_p = float(rng.uniform(0.05, 0.999))
        base = oracle.transform_row(z, T, k, 1.0).probs      # after temperature + top-k
        rd = oracle.transform_row(z, T, k, top_p)
        if rd.top_p_margin < 1e-9:
            continue
        best = None
        for size in range(1, V + 1):
            cands = [s for s in itertools.combinations(range(V), size)
                     if base[list(s)].sum() >= top_p]
            if cands:
                best = max(cands, key=lambda s: base[list(s)].sum())
                break
        assert set(best) == set(np.flatnonzero(rd.probs)), (z, T, k, top_p)
        expect = np.zeros(V)
        expect[list(best)] = base[list(best)]
        np.testing.assert_allclose(rd.probs, expect / expect.sum(), rtol=1e-12, atol=1e-16)
        checked += 1
    assert checked > 250


def test_top_p_one_keeps_everything_and_cut_includes_crossing_token():
    z = np.log(np.array([0.5, 0.3, 0.2]))
    np.testing.assert_allclose(oracle.transform_row(z, 1.0, 0, 1.0).probs, [0.5, 0.3, 0.2])
    # cumulative 0.5, 0.8, 1.0: top_p = 0.6 keeps {0, 1} (the token at which 0.6 is reached)
    np.testing.assert_allclose(oracle.transform_row(z, 1.0, 0, 0.6).probs, [0.625, 0.375, 0.0])
    np.testing.assert_allclose(oracle.transform_row(z, 1.0, 0, 0.4).probs, [1.0, 0.0, 0.0])


def test_banned_tokens_and_row_status():
    z = np.array([0.0, -np.inf, 1.0])
    rd = oracle.transform_row(z, 1.0, 0, 1.0)
    assert rd.probs[1] == 0.0
    np.testing.assert_allclose(rd.probs[[0, 2]], scipy.special.softmax([0.0, 1.0]))
    # top-k larger than the number of finite logits keeps a zero-probability token
    rd = oracle.transform_row(z, 1.0, 2, 1.0)
    assert rd.probs[1] == 0.0
    assert oracle.transform_row(np.full(4, -np.inf), 1.0, 0, 1.0).status == oracle.SEQ_EMPTY_SUPPORT
    assert oracle.transform_row(np.array([0.0, np.nan]), 1.0, 0, 1.0).status == oracle.SEQ_NONFINITE
    assert oracle.transform_row(np.array([0.0, np.inf]), 1.0, 0, 1.0).status == oracle.SEQ_NONFINITE


def test_bf16_widening_matches_torch():
    rng = np.random.default_rng(4)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        ours = oracle.bf16_bits_to_float64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


@pytest.mark.parametrize("T", [0.7, 1.0])
def test_temperature_scales_logits(T):
    z = np.array([2.0, 1.0, 0.0, -3.0])
    np.testing.assert_allclose(oracle.transform_row(z, T, 0, 1.0).probs,
                               scipy.special.softmax(z / T), rtol=1e-13)


def test_top_p_ambiguity_diagnostics():
    """Tokens whose top-p membership turns on a cumulative within 1e-6 of top_p."""
    z = np.log(np.array([0.5, 0.25, 0.25]))
    rd = oracle.transform_row(z, 1.0, 0, 0.75)           # cumulative before token 2 is exactly 0.75
    assert list(rd.ambiguous) == [2] and abs(rd.ambiguous_mass - 0.25) < 1e-12
    rd = oracle.transform_row(z, 1.0, 0, 0.6)
    assert rd.ambiguous.size == 0 and rd.ambiguous_mass == 0.0
    # a dense tail: many tiny tokens around the cut are ambiguous, their mass is tiny
    p = np.concatenate([[0.5], np.full(100000, 0.5 / 100000)])
    rd = oracle.transform_row(np.log(p), 1.0, 0, 0.9)
    assert 0 < rd.ambiguous.size < 1000 and rd.ambiguous_mass < 1e-5
