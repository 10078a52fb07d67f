"""GPU MoE decode with BF16 expert weights (the 16-bit checkpoint variant)
against the oracle, element by element within the layer tolerance."""
import numpy as np
import pytest
import torch

import oracle
from flint_testlib import DeviceLayer, assert_close, flint, combine_terms, margin_x
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu


def _run(dl, x, k, flags=0, bias=None):
    f = flint()
    T, H = x.shape
    ws = dl.workspace(k)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    xc = x.cuda()
    b = bias.cuda() if bias is not None else None
    f.flint_moe_route(xc, dl.router_w, k, ids, w, ws, bias=b, flags=flags)
    f.flint_moe_decode(xc, ids, w, dl.routed, dl.shared, y, ws, flags=flags)
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    return ids.cpu().numpy(), w.cpu().numpy(), synth.bits(y)


def _check(dl, x, k, flags=0, bias=None):
    ids, w, y = _run(dl, x, k, flags, bias)
    rids, rw, ry = oracle.moe_layer(synth.bits(x), synth.bits(dl.L.router_w), k,
                                   bias=None if bias is None else bias.numpy(), **dl.oracle_args())
    for t in range(x.shape[0]):
        assert set(ids[t]) == set(rids[t])
    ref = oracle.moe_experts(synth.bits(x), ids, w, **dl.oracle_args())
    terms = combine_terms(synth.bits(x), rids, rw, dl)
    assert_close(y, ref, "bf16 layer (gpu routing)", terms=terms)
    assert_close(y, ry, "bf16 layer (oracle routing)", terms=terms)
    return y


@pytest.fixture(scope="module")
def small_bf16():
    return DeviceLayer(synth.Layer(21, H=1024, E=16, I=256, I_shared=256, wdtype="bf16"))


@pytest.mark.parametrize("T,k", [(1, 6), (2, 1), (3, 4), (5, 6), (8, 6), (8, 8)])
def test_small_bf16_layer(small_bf16, T, k):
    x = margin_x(synth.bits(small_bf16.L.router_w), T, 1024, k, None, seed=200 + T + 10 * k)
    _check(small_bf16, x, k)


def test_small_bf16_pdl_is_bitwise_identical(small_bf16):
    f = flint()
    x = margin_x(synth.bits(small_bf16.L.router_w), 8, 1024, 6, None, seed=31)
    a = _run(small_bf16, x, 6, flags=0)
    b = _run(small_bf16, x, 6, flags=f.FLINT_PDL)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_bf16_with_tensor_scales():
    """Per-matrix scales given (not all 1): applied to the FP32 sums before rounding."""
    L = synth.Layer(22, H=1024, E=8, I=256, I_shared=256, wdtype="bf16")
    L.ts = synth.tensor_scales(5, (8, 3)) * 25.0
    L.shared["ts"] = synth.tensor_scales(6, (3,)) * 25.0
    dl = DeviceLayer(L)
    x = margin_x(synth.bits(L.router_w), 4, 1024, 2, None, seed=9)
    _check(dl, x, 2)


def test_bf16_without_shared_expert():
    dl = DeviceLayer(synth.Layer(23, H=1024, E=16, I=256, I_shared=0, wdtype="bf16", shared=False))
    x = margin_x(synth.bits(dl.L.router_w), 3, 1024, 6, None, seed=5)
    _check(dl, x, 6)


def test_bf16_wide_shared_expert():
    """Shared expert twice as wide as the routed ones (I_shared = 2 I)."""
    dl = DeviceLayer(synth.Layer(24, H=1024, E=16, I=256, I_shared=512, wdtype="bf16"))
    x = margin_x(synth.bits(dl.L.router_w), 8, 1024, 6, None, seed=6)
    _check(dl, x, 6)


@pytest.fixture(scope="module")
def full_bf16():
    return DeviceLayer(synth.Layer(1001, wdtype="bf16"))


@pytest.mark.parametrize("T", [1, 8])
def test_full_bf16_layer(full_bf16, T):
    f = flint()
    x = margin_x(synth.bits(full_bf16.L.router_w), T, 2048, 6, None, seed=40 + T)
    _check(full_bf16, x, 6, flags=f.FLINT_PDL)


def test_full_bf16_layer_zipf(full_bf16):
    f = flint()
    bias = synth.zipf_bias(77, 256)
    x = margin_x(synth.bits(full_bf16.L.router_w), 8, 2048, 6, bias.numpy(), seed=44)
    _check(full_bf16, x, 6, flags=f.FLINT_PDL, bias=bias)


def test_bf16_rejected_by_one_kernel_layer(small_bf16):
    f = flint()
    ws = small_bf16.workspace(6)
    x = small_bf16.L.x(1).cuda()
    ids = torch.empty((1, 6), dtype=torch.int32, device="cuda")
    w = torch.empty((1, 6), dtype=torch.float32, device="cuda")
    y = torch.empty((1, 1024), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(f.FlintError) as e:
        f.flint_moe_layer(x, small_bf16.router_w, 6, small_bf16.routed, small_bf16.shared, ids, w, y, ws)
    assert e.value.status == f.FLINT_ERR_UNSUPPORTED
