"""Oracle self-tests: the SwiGLU expert and the dense GEMV (CPU only).

Pins: one-hot activations (a GEMV returns one column), a library matmul on
inputs whose double sums are exact, and scipy's expit for SiLU.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from golden_io import same_values
from nvfp4_moe_decode_sigmoid_gb300 import synth


def _exact_x(seed, T, K):
    """bf16 activations k/64, |k| <= 256: every double sum below is exact."""
    rng = np.random.default_rng(seed)
    v = rng.integers(-256, 257, (T, K)).astype(np.float32) / 64.0
    return synth.bits(torch.from_numpy(v).to(torch.bfloat16))


def _onehot(K, c):
    v = np.zeros((1, K), np.float32)
    v[0, c] = 1.0
    return synth.bits(torch.from_numpy(v).to(torch.bfloat16))


def test_dense_gemv_one_hot_returns_a_column():
    N, K = 24, 128
    W = synth.gguf_nvfp4(1, 1, N, K).numpy().reshape(-1)
    dense = oracle.gguf_decode(W, N, K)
    for c in (0, 17, 127):
        y = oracle.dense_gemv(_onehot(K, c), W, N, ts=(0.5,))
        # compared as values: a -0 weight code sums to +0
        assert np.array_equal(oracle.bf16_value(y[0]), oracle.bf16_value(oracle.bf16_round(0.5 * dense[:, c])))


@pytest.mark.parametrize("wdtype", [oracle.W_NVFP4, oracle.W_BF16])
def test_dense_gemv_matches_library_matmul(wdtype):
    N, K, T = 40, 256, 3
    x = _exact_x(2, T, K)
    if wdtype == oracle.W_NVFP4:
        W = synth.gguf_nvfp4(3, 1, N, K).numpy().reshape(-1)
        dense = oracle.gguf_decode(W, N, K)
    else:
        # bf16 weights j/128 keep the sums exact too
        rng = np.random.default_rng(4)
        wf = (rng.integers(-128, 129, (N, K)) / 128.0).astype(np.float32)
        W = synth.bits(torch.from_numpy(wf).to(torch.bfloat16))
        dense = wf.astype(np.float64)
    ref = oracle.bf16_value(x) @ dense.T * 0.25  # power-of-two tensor scale keeps it exact
    y = oracle.dense_gemv(x, W, N, ts=(0.25,), wdtype=wdtype)
    assert same_values(y, oracle.bf16_round(ref))


def test_dense_gemv_swiglu_epilogue():
    N, K, T = 32, 128, 2
    x = _exact_x(5, T, K)
    W = synth.gguf_nvfp4(6, 1, N, K).numpy().reshape(-1)
    dense = oracle.gguf_decode(W, N, K)
    xf = oracle.bf16_value(x)
    g = oracle.bf16_value(oracle.bf16_round(xf @ dense[: N // 2].T * 0.5))
    u = oracle.bf16_value(oracle.bf16_round(xf @ dense[N // 2:].T * 2.0))
    ref = oracle.bf16_round(g * expit(g) * u)
    y = oracle.dense_gemv(x, W, N, ts=(0.5, 2.0), epilogue=oracle.EPI_SWIGLU)
    assert np.array_equal(y, ref)


def test_expert_one_hot_closed_form():
    H, I = 128, 64
    gate = synth.gguf_nvfp4(7, 1, I, H).numpy().reshape(-1)
    up = synth.gguf_nvfp4(8, 1, I, H).numpy().reshape(-1)
    down = synth.gguf_nvfp4(9, 1, H, I).numpy().reshape(-1)
    Wg, Wu, Wd = oracle.gguf_decode(gate, I, H), oracle.gguf_decode(up, I, H), oracle.gguf_decode(down, H, I)
    ts = (0.5, 0.25, 0.125)
    c = 37
    g, u, h, d = oracle.expert(_onehot(H, c)[0], gate, up, down, H, I, ts)
    assert same_values(g, oracle.bf16_round(ts[0] * Wg[:, c]))
    assert same_values(u, oracle.bf16_round(ts[1] * Wu[:, c]))
    gf, uf = oracle.bf16_value(g), oracle.bf16_value(u)
    assert same_values(h, oracle.bf16_round(gf * expit(gf) * uf))
    # h is bf16 and the weights are E2M1 x UE4M3: the double sum is exact
    assert same_values(d, oracle.bf16_round(ts[2] * (Wd @ oracle.bf16_value(h))))


def test_silu_special_values():
    # g = 0 -> h = 0 ; large g -> silu(g) = g to bf16 precision
    H, I = 64, 64
    zero_gate = np.zeros(oracle.gguf_matrix_bytes(I, H), np.uint8)
    up = synth.gguf_nvfp4(10, 1, I, H).numpy().reshape(-1)
    down = synth.gguf_nvfp4(11, 1, H, I).numpy().reshape(-1)
    x = _onehot(H, 3)[0]
    g, u, h, d = oracle.expert(x, zero_gate, up, down, H, I)
    assert not oracle.bf16_value(g).any() and not oracle.bf16_value(h).any() and not oracle.bf16_value(d).any()
    # all gate codes 7 (6.0) with scale 448: g = 2688 for a one-hot x
    big = np.zeros((I * H // 64, 36), np.uint8)
    big[:, :4] = 0x7E
    big[:, 4:] = 0x77
    g, u, h, d = oracle.expert(x, big.reshape(-1), up, down, H, I)
    assert np.all(oracle.bf16_value(g) == 2688.0)
    assert same_values(h, oracle.bf16_round(2688.0 * oracle.bf16_value(u)))
