"""GPU prefill (the MoE layer over many tokens on the tensor cores) against the
oracle: on every token whose top-k margin is at least 1e-3 the selected
experts must match, and on a seeded sample of those tokens the outputs must
be within the layer tolerance. Repeated runs must agree bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from flint_testlib import DeviceLayer, MARGIN, assert_close, bf16_to_f64, layer_flips, flint
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu


def run_prefill(dl, x, k, bias=None):
    f = flint()
    T, H = x.shape
    L = dl.L
    Is = L.Is if L.shared is not None else 0
    ws = torch.empty(f.flint_prefill_workspace_bytes(T, L.E, k, H, L.I, Is), dtype=torch.uint8, device="cuda")
    f.flint_workspace_init(ws)
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    f.flint_moe_prefill(x.cuda(), dl.router_w, k, dl.routed, dl.shared, ids, w, y, ws,
                        bias=None if bias is None else bias.cuda())
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    return ids.cpu().numpy(), w.cpu().numpy(), synth.bits(y)


def check_prefill(dl, x, k, n_sample, bias=None, seed=0):
    ids, w, y = run_prefill(dl, x, k, bias)
    T = x.shape[0]
    xb = synth.bits(x)
    wr = synth.bits(dl.L.router_w)
    b = None if bias is None else bias.numpy()
    rids, rw, s = oracle.router(xb, wr, k, b)
    ss = np.sort(s, axis=1)[:, ::-1]
    margin_ok = (ss[:, k - 1] - ss[:, k] >= MARGIN) if k < s.shape[1] else np.ones(T, bool)
    assert margin_ok.mean() > 0.5
    for t in np.nonzero(margin_ok)[0]:
        assert set(ids[t]) == set(rids[t]), f"token {t}"
        order = np.argsort(ids[t])
        np.testing.assert_allclose(w[t][order], rw[t][np.argsort(rids[t])], rtol=2e-5, atol=1e-7)
    assert np.all((ids >= 0) & (ids < dl.L.E))
    rng = np.random.default_rng(seed)
    cand = np.nonzero(margin_ok)[0]
    pick = np.sort(rng.choice(cand, size=min(n_sample, cand.size), replace=False))
    ref = oracle.moe_experts(xb[pick], rids[pick], rw[pick].astype(np.float32), **dl.oracle_args())
    flips = layer_flips(xb[pick], rids[pick], rw[pick], dl)
    assert_close(y[pick], ref, "prefill", flips=flips)
    return ids, w, y


@pytest.fixture(scope="module")
def small_layer():
    return DeviceLayer(synth.Layer(41, H=1024, E=16, I=256, I_shared=256))


@pytest.mark.parametrize("T,k", [(1, 6), (129, 6), (300, 4), (1000, 6)])
def test_small_prefill(small_layer, T, k):
    x = synth.activations(500 + T, T, 1024)
    check_prefill(small_layer, x, k, n_sample=12, seed=T)


def test_small_prefill_skewed_routing(small_layer):
    """A Zipf bias leaves some experts with no tokens (empty groups)."""
    bias = synth.zipf_bias(9, 16, s=2.0) * 3.0
    x = synth.activations(77, 400, 1024)
    ids, _, _ = check_prefill(small_layer, x, 2, n_sample=16, bias=bias, seed=3)
    assert len(set(ids.reshape(-1).tolist())) < 16


def test_small_prefill_is_deterministic(small_layer):
    x = synth.activations(78, 700, 1024)
    a = run_prefill(small_layer, x, 6)
    b = run_prefill(small_layer, x, 6)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_prefill_without_shared_expert():
    dl = DeviceLayer(synth.Layer(42, H=1024, E=32, I=256, I_shared=0, shared=False))
    x = synth.activations(79, 260, 1024)
    check_prefill(dl, x, 6, n_sample=12, seed=5)


@pytest.fixture(scope="module")
def full_layer():
    return DeviceLayer(synth.Layer(1007))


def test_full_prefill_8k_tokens(full_layer):
    """The prefill workload: 8192 tokens through one full-size layer; ids and
    weights checked on a sample of 512 tokens, outputs on 16 of them."""
    f = flint()
    T, k = 8192, 6
    x = synth.activations(4096, T, 2048)
    ids, w, y = run_prefill(full_layer, x, k)
    rng = np.random.default_rng(11)
    pick = np.sort(rng.choice(T, size=512, replace=False))
    xb = synth.bits(x)[pick]
    rids, rw, s = oracle.router(xb, synth.bits(full_layer.L.router_w), k)
    ss = np.sort(s, axis=1)[:, ::-1]
    ok = ss[:, k - 1] - ss[:, k] >= MARGIN
    for i in np.nonzero(ok)[0]:
        assert set(ids[pick[i]]) == set(rids[i])
    sub = np.nonzero(ok)[0][:16]
    ref = oracle.moe_experts(xb[sub], rids[sub], rw[sub].astype(np.float32), **full_layer.oracle_args())
    flips = layer_flips(xb[sub], rids[sub], rw[sub], full_layer)
    assert_close(y[pick[sub]], ref, "prefill 8k", flips=flips)
    assert np.all(np.isfinite(bf16_to_f64(y)))
    assert np.all((ids >= 0) & (ids < 256))
    del f
