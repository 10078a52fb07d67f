"""Oracle self-tests: sigmoid top-k routing (CPU only).

Pins: logits against a library matmul, scores against scipy's expit,
selection against a brute-force full sort, planted ties, the all-equal
special case and the renormalisation invariant.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from nvfp4_moe_decode_sigmoid_gb300 import synth


def _bits(t):
    return synth.bits(t)


def _brute_topk(scores, k):
    E = scores.shape[0]
    order = sorted(range(E), key=lambda e: (-float(scores[e]), e))
    return order[:k]


@pytest.mark.parametrize("E,k", [(8, 1), (8, 2), (16, 6), (16, 2), (64, 6)])
def test_selection_matches_brute_force(E, k):
    H = 128
    x = _bits(synth.activations(E * 10 + k, 5, H))
    wr = _bits(synth.bf16_normal(E + 3, (E, H), 0.05))
    ids, w, s = oracle.router(x, wr, k)
    for t in range(5):
        assert list(ids[t]) == _brute_topk(s[t], k)
        assert abs(w[t].sum() - 1.0) < 1e-12


def test_scores_match_library_matmul_and_expit():
    E, H, T = 32, 256, 3
    x = _bits(synth.activations(1, T, H))
    wr = _bits(synth.bf16_normal(2, (E, H), 0.02))
    bias = np.linspace(-1, 1, E).astype(np.float32)
    _, _, s = oracle.router(x, wr, 6, bias=bias)
    xf = oracle.bf16_value(x)
    wf = oracle.bf16_value(wr)
    logits = (xf @ wf.T).astype(np.float32) + bias          # FP32 decision precision
    ref = expit(logits.astype(np.float64)).astype(np.float32)
    assert np.array_equal(s, ref)


def test_ties_go_to_lower_index():
    E, H, k = 16, 64, 6
    rng = np.random.default_rng(3)
    wr = np.zeros((E, H), np.float32)
    wr[:, 0] = np.arange(E) * 0.01
    # experts 4, 9 and 13 get the same row as expert 10, the 6th-largest
    # distinct score sits at their value, so only the lowest two of the tie
    # fit: ranks 11..15 are above, then 10 ties with 4, 9, 13.
    wr[[4, 9, 13], :] = wr[10]
    wr[11:, 0] += 1.0
    wr[13, :] = wr[10]
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    xb = _bits(torch.from_numpy(x).to(torch.bfloat16))
    wb = _bits(torch.from_numpy(wr).to(torch.bfloat16))
    ids, w, s = oracle.router(xb, wb, k)
    assert set(ids[0][:4]) == {11, 12, 14, 15}
    assert list(ids[0][4:]) == [4, 9]  # tied with 10 and 13: lower indices win, in index order
    assert list(ids[0]) == _brute_topk(s[0], k)


def test_all_equal_scores():
    E, H, k = 256, 64, 6
    x = _bits(synth.activations(4, 2, H))
    wr = np.zeros((E, H), np.uint16)
    ids, w, s = oracle.router(x, wr, k)
    assert np.all(s == 0.5)
    assert np.array_equal(ids, np.tile(np.arange(k, dtype=np.int32), (2, 1)))
    assert np.allclose(w, 1.0 / k, rtol=0, atol=1e-15)


def test_bias_steers_selection():
    E, H, k = 32, 64, 6
    x = _bits(synth.activations(5, 1, H))
    wr = _bits(synth.bf16_normal(6, (E, H), 0.02))
    bias = np.zeros(E, np.float32)
    bias[[3, 7, 8, 20, 21, 30]] = 10.0
    ids, _, _ = oracle.router(x, wr, k, bias=bias)
    assert set(ids[0]) == {3, 7, 8, 20, 21, 30}


def test_zipf_bias_is_a_distribution():
    b = synth.zipf_bias(1, 256).numpy().astype(np.float64)
    assert abs(np.exp(b).sum() - 1.0) < 1e-5
    assert len(set(np.round(b, 6))) == 256
