"""Oracle self-tests: the whole MoE layer (CPU only).

The layer has no printed worked example, so it is pinned by closed-form
special cases and invariants: identical experts collapse the combine to
2 * d, a zero routed down projection leaves only the shared expert, one
non-zero routed down projection at each rank in turn gives exactly that
rank's weight times its expert's output plus the shared expert (which pins
the pairing of weights with ranks), expert relabelling and token batching
change nothing.
"""
import numpy as np
import pytest

import oracle
from golden_io import same_values
from nvfp4_moe_decode_sigmoid_gb300 import synth

H, E, I, K = 128, 16, 64, 6


def _layer(seed, identical=False):
    gate = synth.gguf_nvfp4(seed + 1, E, I, H).numpy()
    up = synth.gguf_nvfp4(seed + 2, E, I, H).numpy()
    down = synth.gguf_nvfp4(seed + 3, E, H, I).numpy()
    ts = synth.tensor_scales(seed + 4, (E, 3)).numpy()
    sh = dict(gate=synth.gguf_nvfp4(seed + 5, 1, I, H).numpy(), up=synth.gguf_nvfp4(seed + 6, 1, I, H).numpy(),
              down=synth.gguf_nvfp4(seed + 7, 1, H, I).numpy(), ts=synth.tensor_scales(seed + 8, (3,)).numpy(), I=I)
    if identical:
        gate[:] = sh["gate"][0]
        up[:] = sh["up"][0]
        down[:] = sh["down"][0]
        ts[:] = sh["ts"]
    wr = synth.bits(synth.bf16_normal(seed + 9, (E, H), 0.05))
    return gate, up, down, ts, sh, wr


def test_identical_experts_collapse_to_twice_the_expert():
    gate, up, down, ts, sh, wr = _layer(10, identical=True)
    x = synth.bits(synth.activations(1, 3, H))
    ids, w, y = oracle.moe_layer(x, wr, K, E, I, gate, up, down, ts, shared=sh)
    for t in range(3):
        _, _, _, d = oracle.expert(x[t], sh["gate"], sh["up"], sh["down"], H, I, sh["ts"])
        assert same_values(y[t], oracle.bf16_round(2.0 * oracle.bf16_value(d)))
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)


def test_zero_routed_down_leaves_the_shared_expert():
    gate, up, down, ts, sh, wr = _layer(20)
    down[:] = 0
    x = synth.bits(synth.activations(2, 2, H))
    _, _, y = oracle.moe_layer(x, wr, K, E, I, gate, up, down, ts, shared=sh)
    for t in range(2):
        _, _, _, d = oracle.expert(x[t], sh["gate"], sh["up"], sh["down"], H, I, sh["ts"])
        assert same_values(y[t], d)


def test_single_routed_expert_without_shared_is_that_expert():
    gate, up, down, ts, _, wr = _layer(30)
    x = synth.bits(synth.activations(3, 1, H))
    ids, w, y = oracle.moe_layer(x, wr, 1, E, I, gate, up, down, ts, shared=None)
    e = int(ids[0, 0])
    assert w[0, 0] == 1.0
    _, _, _, d = oracle.expert(x[0], gate[e], up[e], down[e], H, I, ts[e])
    assert same_values(y[0], d)


def test_expert_relabelling_is_invisible():
    gate, up, down, ts, sh, wr = _layer(40)
    x = synth.bits(synth.activations(4, 2, H))
    ids, w, y = oracle.moe_layer(x, wr, K, E, I, gate, up, down, ts, shared=sh)
    perm = np.random.default_rng(0).permutation(E)
    inv = np.argsort(perm)
    ids2, w2, y2 = oracle.moe_layer(x, wr[perm], K, E, I, gate[perm], up[perm], down[perm], ts[perm], shared=sh)
    assert np.array_equal(y, y2)
    assert np.array_equal(np.sort(inv[ids], axis=1), np.sort(ids2, axis=1))


def test_tokens_are_independent():
    gate, up, down, ts, sh, wr = _layer(50)
    x = synth.bits(synth.activations(5, 4, H))
    _, _, y = oracle.moe_layer(x, wr, K, E, I, gate, up, down, ts, shared=sh)
    for t in range(4):
        _, _, y1 = oracle.moe_layer(x[t:t + 1], wr, K, E, I, gate, up, down, ts, shared=sh)
        assert np.array_equal(y[t], y1[0])


def test_bf16_weight_variant_identical_experts():
    gate = np.repeat(synth.bits(synth.bf16_normal(1, (1, I, H), 0.02)), E, axis=0)
    up = np.repeat(synth.bits(synth.bf16_normal(2, (1, I, H), 0.02)), E, axis=0)
    down = np.repeat(synth.bits(synth.bf16_normal(3, (1, H, I), 0.02)), E, axis=0)
    wr = synth.bits(synth.bf16_normal(4, (E, H), 0.05))
    x = synth.bits(synth.activations(6, 2, H))
    sh = dict(gate=gate[:1], up=up[:1], down=down[:1], ts=None, I=I)
    _, _, y = oracle.moe_layer(x, wr, K, E, I, gate, up, down, None, shared=sh, wdtype=oracle.W_BF16)
    for t in range(2):
        _, _, _, d = oracle.expert(x[t], gate[0], up[0], down[0], H, I, wdtype=oracle.W_BF16)
        assert same_values(y[t], oracle.bf16_round(2.0 * oracle.bf16_value(d)))


def _f32(v):
    return np.asarray(v, np.float64).astype(np.float32)


@pytest.mark.parametrize("k", [2, 6])
def test_one_live_expert_per_rank_pins_the_weight_of_each_rank(k):
    """All routed down matrices are zero except that of the expert at rank r,
    so y = bf16(fl(w_r d_r) + d_shared) in FP32 (the other ranks add exact
    zeros). Distinct weights per rank: giving rank r another rank's weight,
    or the weights in reverse order, changes y."""
    gate, up, down, ts, sh, _ = _layer(60)
    x = synth.bits(synth.activations(7, 1, H))
    ids = np.array([[3, 11, 5, 0, 14, 8][:k]], np.int32)
    w = _f32(np.linspace(0.9, 0.1, k) / np.linspace(0.9, 0.1, k).sum())[None, :]
    assert len(set(w[0].tolist())) == k
    _, _, _, d_s = oracle.expert(x[0], sh["gate"], sh["up"], sh["down"], H, I, sh["ts"])
    ds = oracle.bf16_value(d_s)
    for r in range(k):
        e = int(ids[0, r])
        live = np.zeros_like(down)
        live[e] = down[e]
        y = oracle.moe_experts(x, ids, w, E, I, gate, up, live, ts, shared=sh)
        _, _, _, d = oracle.expert(x[0], gate[e], up[e], down[e], H, I, ts[e])
        dv = oracle.bf16_value(d)
        assert np.any(dv != 0)
        term = (np.float64(w[0, r]) * dv).astype(np.float32)        # fmaf(w, d, 0): one rounding
        expect = oracle.bf16_round((term + _f32(ds)).astype(np.float32).astype(np.float64))
        assert same_values(y[0], expect), f"rank {r}"
        # another rank's weight would give a different output
        other = (np.float64(w[0, (r + 1) % k]) * dv).astype(np.float32)
        wrong = oracle.bf16_round((other + _f32(ds)).astype(np.float32).astype(np.float64))
        assert not same_values(wrong, expect)


def test_openmp_build_gives_the_same_bits():
    """The OpenMP build of the oracle (output rows split over threads, each
    row summed in index order by one thread) returns exactly what the plain
    build returns."""
    gate, up, down, ts, sh, wr = _layer(70)
    x = synth.bits(synth.activations(8, 3, H))
    ref = oracle.moe_layer(x, wr, K, E, I, gate, up, down, ts, shared=sh)
    try:
        if oracle.use_openmp(4) == 0:
            pytest.skip("no OpenMP compiler here")
        got = oracle.moe_layer(x, wr, K, E, I, gate, up, down, ts, shared=sh)
    finally:
        oracle.use_openmp(-1)
    for a, b in zip(ref, got):
        assert np.array_equal(a, b)
