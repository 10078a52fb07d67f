"""Oracle self-tests: the whole MoE layer (CPU only).

The layer has no printed worked example, so it is pinned by closed-form
special cases and invariants: identical experts collapse the combine to
2 * d, a zero routed down projection leaves only the shared expert, expert
relabelling and token batching change nothing.
"""
import numpy as np

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
