"""The fused layer kernel (flint_moe_layer: routing, gate/up, down and combine
in one cooperative launch) against the oracle: selection bit-exact, weights
to FP32 rounding, y within the layer tolerance."""
import numpy as np
import pytest
import torch

import oracle
from flint_testlib import DeviceLayer, assert_close, flint, combine_terms, margin_x
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu


def _run(dl, x, k, bias=None, flags=0, ws=None):
    f = flint()
    T, H = x.shape
    ws = dl.workspace(k) if ws is None else ws
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    b = bias.cuda() if bias is not None else None
    f.flint_moe_layer(x.cuda(), dl.router_w, k, dl.routed, dl.shared, ids, w, y, ws, bias=b, flags=flags)
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    return ids.cpu().numpy(), w.cpu().numpy(), synth.bits(y)


def _check(dl, x, k, bias=None, flags=0):
    ids, w, y = _run(dl, x, k, bias, flags)
    rids, rw, ry = oracle.moe_layer(synth.bits(x), synth.bits(dl.L.router_w), k,
                                    bias=None if bias is None else bias.numpy(), **dl.oracle_args())
    assert np.array_equal(ids, rids), f"selection differs: {ids} vs {rids}"
    assert np.allclose(w, rw, rtol=2e-6, atol=1e-7), f"weights differ: {w} vs {rw}"
    ref = oracle.moe_experts(synth.bits(x), ids, w, **dl.oracle_args())
    terms = combine_terms(synth.bits(x), rids, rw, dl)
    assert_close(y, ref, "fused layer (gpu routing)", terms=terms)
    assert_close(y, ry, "fused layer (oracle routing)", terms=terms)
    return ids, w, y


@pytest.fixture(scope="module")
def small_layer():
    return DeviceLayer(synth.Layer(11, H=1024, E=16, I=256, I_shared=256))


@pytest.mark.parametrize("T,k", [(1, 6), (2, 1), (5, 4), (8, 6), (8, 8)])
def test_small_layer(small_layer, T, k):
    x = margin_x(synth.bits(small_layer.L.router_w), T, 1024, k, None, seed=T + 10 * k)
    _check(small_layer, x, k)


def test_small_layer_with_bias_and_pdl(small_layer):
    f = flint()
    bias = synth.zipf_bias(5, 16)
    x = margin_x(synth.bits(small_layer.L.router_w), 6, 1024, 6, bias.numpy(), seed=31)
    _check(small_layer, x, 6, bias=bias, flags=f.FLINT_PDL)


def test_without_shared_expert():
    dl = DeviceLayer(synth.Layer(12, H=1024, E=16, I=256, I_shared=0, shared=False))
    x = margin_x(synth.bits(dl.L.router_w), 3, 1024, 6, None, seed=4)
    _check(dl, x, 6)


def test_shared_expert_wider_than_routed():
    dl = DeviceLayer(synth.Layer(13, H=1024, E=16, I=256, I_shared=1024))
    x = margin_x(synth.bits(dl.L.router_w), 4, 1024, 6, None, seed=5)
    _check(dl, x, 6)


def test_many_experts_wide_topk():
    # E above 256: the top-k warp takes 32 scores per lane
    dl = DeviceLayer(synth.Layer(14, H=1024, E=600, I=256, I_shared=256))
    x = margin_x(synth.bits(dl.L.router_w), 3, 1024, 8, None, seed=6)
    _check(dl, x, 8)


@pytest.mark.parametrize("case", ["no_shared", "wide_shared", "many_experts_k8", "bias"])
def test_one_token_shapes(case):
    """One token runs the one-token kernel (equal shares of every step per
    CTA): without a shared expert, with a shared expert wider than the routed
    ones, with E = 600 (fewer than one router row per CTA on some, top-k over
    32 scores per lane) and k = 8, and with a router bias."""
    f = flint()
    k, bias = 6, None
    if case == "no_shared":
        dl = DeviceLayer(synth.Layer(12, H=1024, E=16, I=256, I_shared=0, shared=False))
    elif case == "wide_shared":
        dl = DeviceLayer(synth.Layer(13, H=1024, E=16, I=256, I_shared=1024))
    elif case == "many_experts_k8":
        dl, k = DeviceLayer(synth.Layer(14, H=1024, E=600, I=256, I_shared=256)), 8
    else:
        dl = DeviceLayer(synth.Layer(15, H=2048, E=256, I=512, I_shared=512))
        bias = synth.zipf_bias(5, 256)
    H = dl.L.router_w.shape[1]
    x = margin_x(synth.bits(dl.L.router_w), 1, H, k, None if bias is None else bias.numpy(), seed=50)
    _check(dl, x, k, bias=bias, flags=f.FLINT_PDL)


@pytest.fixture(scope="module")
def full_layer():
    return DeviceLayer(synth.Layer(1000, H=2048, E=256, I=512, I_shared=512))


def test_full_layer_batch1(full_layer):
    f = flint()
    x = margin_x(synth.bits(full_layer.L.router_w), 1, 2048, 6, None, seed=7)
    _check(full_layer, x, 6, flags=f.FLINT_PDL)


def test_full_layer_batch8_uniform(full_layer):
    x = margin_x(synth.bits(full_layer.L.router_w), 8, 2048, 6, None, seed=8)
    _check(full_layer, x, 6)


@pytest.mark.parametrize("T", [2, 3, 4, 6, 7])
def test_full_layer_other_batches(full_layer, T):
    """Batches around the switch from prefetched down rows (T <= 3) to the down
    ring (T >= 4), with the routed gate/up pairs dealt over all CTAs."""
    x = margin_x(synth.bits(full_layer.L.router_w), T, 2048, 6, None, seed=40 + T)
    _check(full_layer, x, 6)


def test_full_layer_batch8_zipf(full_layer):
    f = flint()
    bias = synth.zipf_bias(3, 256)
    x = margin_x(synth.bits(full_layer.L.router_w), 8, 2048, 6, bias.numpy(), seed=9)
    _check(full_layer, x, 6, bias=bias, flags=f.FLINT_PDL)


@pytest.mark.parametrize("T", [1, 8])
def test_repeated_calls_on_one_workspace_are_deterministic(full_layer, T):
    # the exchange counts are back at zero after every call
    x = margin_x(synth.bits(full_layer.L.router_w), T, 2048, 6, None, seed=10)
    ws = full_layer.workspace(6)
    outs = [_run(full_layer, x, 6, ws=ws) for _ in range(4)]
    for o in outs[1:]:
        for u, v in zip(o, outs[0]):
            assert np.array_equal(u, v)


def test_matches_the_three_kernel_path(full_layer):
    f = flint()
    x = margin_x(synth.bits(full_layer.L.router_w), 8, 2048, 6, None, seed=12)
    ids, w, y = _run(full_layer, x, 6)
    ws = full_layer.workspace(6)
    ids2 = torch.empty((8, 6), dtype=torch.int32, device="cuda")
    w2 = torch.empty((8, 6), dtype=torch.float32, device="cuda")
    y2 = torch.empty((8, 2048), dtype=torch.bfloat16, device="cuda")
    xc = x.cuda()
    f.flint_moe_route(xc, full_layer.router_w, 6, ids2, w2, ws)
    f.flint_moe_decode(xc, ids2, w2, full_layer.routed, full_layer.shared, y2, ws)
    assert np.array_equal(ids, ids2.cpu().numpy())
    assert np.allclose(w, w2.cpu().numpy(), rtol=2e-6, atol=1e-7)
    assert_close(y, synth.bits(y2), "fused vs three kernels", terms=combine_terms(synth.bits(x), ids, w, full_layer))


def test_pdl_chained_layers_in_a_graph_match_single_calls(full_layer):
    """Several layer calls PDL-chained on one stream and on one workspace,
    captured in a CUDA graph and replayed (each call may start while the
    previous one finishes; the call counter gives each its own tag), give the
    same bits as the same calls made one at a time with a synchronisation in
    between."""
    f = flint()
    k, T = 6, 8
    xs = [margin_x(synth.bits(full_layer.L.router_w), T, 2048, k, None, seed=80 + i).cuda() for i in range(3)]
    ws = full_layer.workspace(k)
    outs = [(torch.empty((T, k), dtype=torch.int32, device="cuda"), torch.empty((T, k), dtype=torch.float32,
                                                                                  device="cuda"),
             torch.empty((T, 2048), dtype=torch.bfloat16, device="cuda")) for _ in range(6)]
    steps = [(xs[i % 3], (T if i % 2 == 0 else 1)) for i in range(6)]

    def run(flags):
        for (x, t), (ids, w, y) in zip(steps, outs):
            f.flint_moe_layer(x[:t], full_layer.router_w, k, full_layer.routed, full_layer.shared, ids[:t], w[:t],
                              y[:t], ws, flags=flags)

    ref = []
    for (x, t), (ids, w, y) in zip(steps, outs):
        f.flint_moe_layer(x[:t], full_layer.router_w, k, full_layer.routed, full_layer.shared, ids[:t], w[:t], y[:t],
                          ws)
        torch.cuda.synchronize()
        ref.append((ids[:t].clone(), w[:t].clone(), y[:t].clone()))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        run(f.FLINT_PDL)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run(f.FLINT_PDL)
        for (_, _, y) in outs:
            y.zero_()
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    for (x, t), (ids, w, y), (ri, rw, ry) in zip(steps, outs, ref):
        assert torch.equal(ids[:t], ri) and torch.equal(w[:t], rw)
        assert torch.equal(y[:t].view(torch.int16), ry.view(torch.int16))


@pytest.mark.parametrize("T", [1, 3])
def test_next_layer_prefetch_changes_nothing(full_layer, T):
    """flint_moe_layer with the next layer's ranges to pull into L2 (here
    another layer's router and shared expert, and the ranges at any offset of
    16 bytes) gives the same bits as without."""
    f = flint()
    other = DeviceLayer(synth.Layer(1008))
    x = margin_x(synth.bits(full_layer.L.router_w), T, 2048, 6, None, seed=21)
    base = _run(full_layer, x, 6)
    nxt = f.l2_prefetch(other.router_w, other.shared.gate_up[16:], other.shared.down[: 4096 * 16])
    ids = torch.empty((T, 6), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 6), dtype=torch.float32, device="cuda")
    y = torch.empty((T, 2048), dtype=torch.bfloat16, device="cuda")
    ws = full_layer.workspace(6)
    f.flint_moe_layer(x.cuda(), full_layer.router_w, 6, full_layer.routed, full_layer.shared, ids, w, y, ws,
                      flags=f.FLINT_PDL, next=nxt)
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    for u, v in zip((ids.cpu().numpy(), w.cpu().numpy(), synth.bits(y)), base):
        assert np.array_equal(u, v)

