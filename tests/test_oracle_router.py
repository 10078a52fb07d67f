"""Oracle self-tests: sigmoid top-k routing (CPU only).

Pins: logits against an FP32 running sum written out in numpy (each step one
float32 rounding; the products of two bf16 values are exact in float32) and
against a library matmul, scores against scipy's expit of those logits,
selection against a brute-force full sort, planted ties, the all-equal
special case and the renormalisation invariant (weights are FP32: they sum to
1 within the rounding of k float32 steps).
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
        assert abs(w[t].sum() - 1.0) < 4 * k * 2.0 ** -24
        # weight j belongs to the expert of rank j: its score over the FP32 sum of the selected scores
        sel = s[t][ids[t]]
        tot = np.float32(0)
        for v in sel:
            tot = np.float32(tot + v)
        assert np.array_equal(w[t].astype(np.float32), (sel / tot).astype(np.float32))


def test_scores_match_library_matmul_and_expit():
    E, H, T = 32, 256, 3
    x = _bits(synth.activations(1, T, H))
    wr = _bits(synth.bf16_normal(2, (E, H), 0.02))
    bias = np.linspace(-1, 1, E).astype(np.float32)
    _, _, s = oracle.router(x, wr, 6, bias=bias)
    xf = oracle.bf16_value(x)
    wf = oracle.bf16_value(wr)
    # FP32 running sums in index order: products exact in float32, one rounding per add
    acc = np.zeros((T, E), np.float32)
    for h in range(H):
        acc = (acc + np.outer(xf[:, h], wf[:, h]).astype(np.float32)).astype(np.float32)
    exact = xf @ wf.T
    assert np.all(np.abs(acc - exact) <= H * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf).T))
    logits = (acc + bias).astype(np.float32)
    ref = expit(logits.astype(np.float64))
    # the FP32 sigmoid is within 2 float32 ulps of the exact value of the FP32 logit
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(s.astype(np.float64) - ref) <= 2 * ulp)


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
    assert np.allclose(w, 1.0 / k, rtol=0, atol=2.0 ** -24)


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
