"""Pins of the oracle's residual add + RMSNorm and of its decode-stack
composition, against closed forms and invariants that the mathematics fixes
(not a retyping of the oracle's own formula)."""
import numpy as np
import pytest

import oracle


def bits(v):
    return oracle.bf16_round(np.asarray(v, np.float64))


def val(b):
    return oracle.bf16_value(b)


@pytest.mark.parametrize("c", [0.375, -3.0, 1e-3, 96.0])
def test_constant_vector_normalises_to_one(c):
    # mean(r^2) = c^2, so r / sqrt(mean) = sign(c) exactly when eps = 0
    r = bits(np.full((2, 64), c))
    _, x = oracle.residual_rmsnorm(r, None, None, eps=0.0)
    assert np.all(val(x) == np.sign(c))


def test_single_spike_uses_the_mean_not_the_sum():
    # one nonzero c among H = 16: mean = c^2 / 16, so x = 4 sign(c) there and 0 elsewhere
    r = np.zeros((1, 16))
    r[0, 5] = -2.5
    _, x = oracle.residual_rmsnorm(bits(r), None, None, eps=0.0)
    expect = np.zeros(16)
    expect[5] = -4.0
    assert np.array_equal(val(x)[0], expect)


def test_eps_equal_to_the_mean_square():
    # r = c everywhere and eps = c^2: x = 1 / sqrt(2), whose bf16 rounding is 181 / 256
    r = bits(np.full((1, 32), 0.5))
    _, x = oracle.residual_rmsnorm(r, None, None, eps=0.25)
    assert np.all(val(x) == 181.0 / 256.0)


def test_power_of_two_scaling_is_invisible():
    rng = np.random.default_rng(3)
    r = bits(rng.normal(size=(3, 256)))
    _, x1 = oracle.residual_rmsnorm(r, None, None, eps=0.0)
    _, x2 = oracle.residual_rmsnorm(bits(val(r) * 8.0), None, None, eps=0.0)
    _, x3 = oracle.residual_rmsnorm(bits(val(r) / 1024.0), None, None, eps=0.0)
    assert np.array_equal(x1, x2) and np.array_equal(x1, x3)


def test_gamma_scales_elementwise():
    rng = np.random.default_rng(4)
    r = bits(rng.normal(size=(2, 64)))
    _, x = oracle.residual_rmsnorm(r, None, None, eps=1e-6)
    g = np.tile(np.array([1.0, 2.0, 4.0, 0.5]), 16)
    _, xg = oracle.residual_rmsnorm(r, None, bits(g), eps=1e-6)
    assert np.array_equal(val(xg), val(x) * g)  # powers of two: exact


def test_unit_mean_square():
    rng = np.random.default_rng(5)
    r = bits(rng.normal(size=(4, 2048)) * 7.0)
    _, x = oracle.residual_rmsnorm(r, None, None, eps=1e-6)
    ms = (val(x) ** 2).mean(axis=1)
    assert np.all(np.abs(ms - 1.0) < 4e-3)  # bf16 rounding of each element: relative error <= 2^-9


def test_residual_cancels_to_zero():
    rng = np.random.default_rng(6)
    r = bits(rng.normal(size=(2, 128)))
    neg = bits(-val(r))
    r_out, x = oracle.residual_rmsnorm(r, neg, None, eps=1e-6)
    assert np.all(val(r_out) == 0.0) and np.all(val(x) == 0.0)


@pytest.mark.parametrize("r0,y,expect", [
    (1.0, 2.0 ** -9, 1.0),                        # below half an ulp (2^-8 at 1.0)
    (1.0, 3 * 2.0 ** -9, 1.0 + 2.0 ** -7),        # above half an ulp
    (1.0, 2.0 ** -8, 1.0),                        # tie, even mantissa stays
    (1.0 + 2.0 ** -7, 2.0 ** -8, 1.0 + 2.0 ** -6),  # tie, odd mantissa rounds up
    (-3.0, 3.0 + 2.0 ** -6, 2.0 ** -6),           # cancellation is exact
])
def test_residual_add_rounds_to_nearest_even(r0, y, expect):
    r_out, _ = oracle.residual_rmsnorm(bits([[r0] * 8]), bits([[y] * 8]), None, eps=1e-6)
    assert np.all(val(r_out) == expect)


def test_stack_of_zero_blocks_only_normalises():
    """With every block's output zero (all-zero weights), the residual stream
    keeps the input exactly and each block sees rmsnorm(x0)."""
    H, F, E, I = 1024, 1024, 8, 256
    rng = np.random.default_rng(7)
    x0 = bits(rng.normal(size=(2, H)))
    zero_gguf = lambda rows, cols: np.zeros(oracle.gguf_matrix_bytes(rows, cols), np.uint8)  # noqa: E731
    dense = dict(kind="dense", F=F, gate_up=zero_gguf(2 * F, H), ts_gu=(1.0, 1.0), down=zero_gguf(H, F),
                 ts_down=(1.0,))
    moe = dict(kind="moe", wr=bits(rng.normal(size=(E, H)) * 0.02), k=2, E=E, I=I,
               gate=np.zeros(E * oracle.gguf_matrix_bytes(I, H), np.uint8),
               up=np.zeros(E * oracle.gguf_matrix_bytes(I, H), np.uint8),
               down=np.zeros(E * oracle.gguf_matrix_bytes(H, I), np.uint8), ts=np.ones((E, 3), np.float32))
    r, trace, ids = oracle.decode_stack(x0, [dense, moe, moe])
    assert np.array_equal(r, x0)
    _, xn = oracle.residual_rmsnorm(x0, None, None, 1e-6)
    for x, y in trace:
        assert np.array_equal(x, xn) and np.all(val(y) == 0.0)
    assert len(ids) == 2 and ids[0].shape == (2, 2)
