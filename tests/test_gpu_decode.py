"""GPU MoE decode (gate/up + SiLU, down + combine) and the whole layer against
the oracle, element by element within the layer tolerance."""
import numpy as np
import pytest
import torch

import oracle
from flint_testlib import DeviceLayer, assert_close, flint, combine_terms, margin_x
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu


def _layer_run(dl, x, k, bias=None, flags=0, route_flags=None):
    f = flint()
    T, H = x.shape
    ws = dl.workspace(k)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    xc = x.cuda()
    b = bias.cuda() if bias is not None else None
    f.flint_moe_route(xc, dl.router_w, k, ids, w, ws, bias=b, flags=flags if route_flags is None else route_flags)
    f.flint_moe_decode(xc, ids, w, dl.routed, dl.shared, y, ws, flags=flags)
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    return ids.cpu().numpy(), w.cpu().numpy(), synth.bits(y)


def _check_layer(dl, x, k, bias=None, flags=0):
    ids, w, y = _layer_run(dl, x, k, bias, flags)
    rids, rw, ry = oracle.moe_layer(synth.bits(x), synth.bits(dl.L.router_w), k,
                                    bias=None if bias is None else bias.numpy(), **dl.oracle_args())
    for t in range(x.shape[0]):
        assert set(ids[t]) == set(rids[t])
    # the experts' outputs given the GPU's own routing (same ids, its weights)
    ref = oracle.moe_experts(synth.bits(x), ids, w, **dl.oracle_args())
    terms = combine_terms(synth.bits(x), rids, rw, dl)
    assert_close(y, ref, "layer (gpu routing)", terms=terms)
    assert_close(y, ry, "layer (oracle routing)", terms=terms)
    return y


@pytest.fixture(scope="module")
def small_layer():
    return DeviceLayer(synth.Layer(11, H=1024, E=16, I=256, I_shared=256))


@pytest.mark.parametrize("T,k", [(1, 6), (2, 1), (5, 4), (8, 6), (8, 8)])
def test_small_layer(small_layer, T, k):
    x = margin_x(synth.bits(small_layer.L.router_w), T, 1024, k, None, seed=T + 10 * k)
    _check_layer(small_layer, x, k)


def test_small_layer_pdl_is_bitwise_identical(small_layer):
    f = flint()
    x = margin_x(synth.bits(small_layer.L.router_w), 8, 1024, 6, None, seed=3)
    a = _layer_run(small_layer, x, 6, flags=0)
    b = _layer_run(small_layer, x, 6, flags=f.FLINT_PDL)
    c = _layer_run(small_layer, x, 6, flags=f.FLINT_PDL | f.FLINT_PDL_AFTER_ROUTE, route_flags=f.FLINT_PDL)
    for u, v, w in zip(a, b, c):
        assert np.array_equal(u, v) and np.array_equal(u, w)


def test_without_shared_expert():
    dl = DeviceLayer(synth.Layer(12, H=1024, E=16, I=256, I_shared=0, shared=False))
    x = margin_x(synth.bits(dl.L.router_w), 3, 1024, 6, None, seed=4)
    _check_layer(dl, x, 6)


def test_shared_expert_wider_than_routed():
    dl = DeviceLayer(synth.Layer(13, H=1024, E=16, I=256, I_shared=1024))
    x = margin_x(synth.bits(dl.L.router_w), 4, 1024, 6, None, seed=5)
    _check_layer(dl, x, 6)


def _decode_ws(dl, k, path):
    """A workspace for flint_moe_decode: sized with the experts' hidden size
    (one cooperative kernel) or with hidden 0 (the two-kernel path)."""
    if path == "one kernel":
        return dl.workspace(k)
    f = flint()
    Is = dl.L.Is if dl.L.shared is not None else 0
    ws = torch.empty(f.flint_workspace_bytes(dl.L.E, k, 0, dl.L.I, Is), dtype=torch.uint8, device="cuda")
    f.flint_workspace_init(ws)
    return ws


PATHS = ["one kernel", "two kernels"]

# hand-made routings: an expert picked twice by one token, experts shared
# between tokens; one token (the one-kernel path splits down by output rows)
# and several (split by expert)
REPEATED = {
    1: ([[3, 3, 7, 0]], [[0.4, 0.3, 0.2, 0.1]]),
    3: ([[3, 3, 7, 0], [7, 0, 15, 3], [15, 14, 13, 12]],
        [[0.4, 0.3, 0.2, 0.1], [0.25, 0.25, 0.25, 0.25], [0.7, 0.1, 0.1, 0.1]]),
    8: ([[5, 5, 5, 5]] + [[(3 * t + j) % 16 for j in range(4)] for t in range(1, 8)],
        [[0.1, 0.2, 0.3, 0.4]] * 8),
}


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T", sorted(REPEATED))
def test_decode_with_repeated_and_shared_ids(small_layer, T, path):
    f = flint()
    dl = small_layer
    k, H = 4, 1024
    x = synth.activations(21 + T, T, H)
    ids = np.array(REPEATED[T][0], np.int32)
    w = np.array(REPEATED[T][1], np.float32)
    ws = _decode_ws(dl, k, path)
    y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    f.flint_moe_decode(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), dl.routed, dl.shared, y,
                       ws)
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    ref = oracle.moe_experts(synth.bits(x), ids, w, **dl.oracle_args())
    assert_close(synth.bits(y), ref, f"repeated ids ({path})", terms=combine_terms(synth.bits(x), ids, w, dl))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T", [1, 3])
def test_out_of_range_id_is_reported_and_adds_nothing(small_layer, T, path):
    """An id outside [0, E) is reported (FLINT_ERR_INVALID_ARG from the check,
    which clears it), its weights are never read against any expert, and y is
    the combine of the other ranks: the oracle with that rank's weight 0."""
    f = flint()
    dl = small_layer
    k, H = 2, 1024
    ids = np.array([[1, 999], [-4, 2], [6, 5]][:T], np.int32)
    w = np.array([[0.5, 0.5], [0.5, 0.5], [0.6, 0.4]][:T], np.float32)
    x = synth.activations(2 + T, T, H)
    ws = _decode_ws(dl, k, path)
    y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    f.flint_moe_decode(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), dl.routed, dl.shared, y,
                       ws)
    assert f.flint_workspace_check(ws) == f.FLINT_ERR_INVALID_ARG
    assert f.flint_workspace_check(ws) == f.FLINT_OK  # cleared
    bad = (ids < 0) | (ids >= dl.L.E)
    ids_ref, w_ref = np.where(bad, 0, ids).astype(np.int32), np.where(bad, 0.0, w).astype(np.float32)
    ref = oracle.moe_experts(synth.bits(x), ids_ref, w_ref, **dl.oracle_args())
    assert_close(synth.bits(y), ref, f"invalid id ({path})", terms=combine_terms(synth.bits(x), ids_ref, w_ref, dl))


@pytest.mark.parametrize("T", [1, 8])
def test_decode_paths_agree_with_the_oracle_on_router_output(T):
    """The one-kernel and the two-kernel decode on the router's own ids and
    weights (full Flint shape): each within the tolerance of the oracle, and
    each deterministic."""
    f = flint()
    dl = _full()
    k, H = 6, 2048
    x = margin_x(synth.bits(dl.L.router_w), T, H, k, None, seed=40 + T)
    xc = x.cuda()
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    f.flint_moe_route(xc, dl.router_w, k, ids, w, dl.workspace(k))
    ref = oracle.moe_experts(synth.bits(x), ids.cpu().numpy(), w.cpu().numpy(), **dl.oracle_args())
    terms = combine_terms(synth.bits(x), ids.cpu().numpy(), w.cpu().numpy(), dl)
    for path in PATHS:
        ws = _decode_ws(dl, k, path)
        outs = []
        for _ in range(2):
            y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
            f.flint_moe_decode(xc, ids, w, dl.routed, dl.shared, y, ws, flags=f.FLINT_PDL)
            assert f.flint_workspace_check(ws) == f.FLINT_OK
            outs.append(synth.bits(y))
        assert np.array_equal(outs[0], outs[1]), path
        assert_close(outs[0], ref, f"decode ({path})", terms=terms)


_FULL = {}


def _full():
    # one Flint-shaped layer: H 2048, 256 routed + 1 shared expert, I 512
    if "dl" not in _FULL:
        _FULL["dl"] = DeviceLayer(synth.Layer(1000, H=2048, E=256, I=512, I_shared=512))
    return _FULL["dl"]


@pytest.fixture(scope="module")
def full_layer():
    return _full()


def test_full_layer_batch1(full_layer):
    f = flint()
    x = margin_x(synth.bits(full_layer.L.router_w), 1, 2048, 6, None, seed=7)
    _check_layer(full_layer, x, 6, flags=f.FLINT_PDL)


def test_full_layer_batch1_after_route(full_layer):
    f = flint()
    x = margin_x(synth.bits(full_layer.L.router_w), 1, 2048, 6, None, seed=17)
    ids, w, y = _layer_run(full_layer, x, 6, flags=f.FLINT_PDL | f.FLINT_PDL_AFTER_ROUTE, route_flags=f.FLINT_PDL)
    ref = oracle.moe_experts(synth.bits(x), ids, w, **full_layer.oracle_args())
    assert_close(y, ref, "layer (x staged before the wait)", terms=combine_terms(synth.bits(x), ids, w, full_layer))


def test_full_layer_batch8_uniform(full_layer):
    f = flint()
    x = margin_x(synth.bits(full_layer.L.router_w), 8, 2048, 6, None, seed=8)
    _check_layer(full_layer, x, 6, flags=f.FLINT_PDL | f.FLINT_PDL_AFTER_ROUTE)


def test_full_layer_batch8_zipf(full_layer):
    f = flint()
    bias = synth.zipf_bias(3, 256)
    x = margin_x(synth.bits(full_layer.L.router_w), 8, 2048, 6, bias.numpy(), seed=9)
    _check_layer(full_layer, x, 6, bias=bias, flags=f.FLINT_PDL)


def test_full_layer_is_deterministic(full_layer):
    f = flint()
    x = margin_x(synth.bits(full_layer.L.router_w), 8, 2048, 6, None, seed=10)
    outs = [_layer_run(full_layer, x, 6, flags=f.FLINT_PDL)[2] for _ in range(3)]
    assert all(np.array_equal(o, outs[0]) for o in outs)
