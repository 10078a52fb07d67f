"""Host-buffer paths of the fused layer give the device path's bits: x copied
in from pinned host memory on a side stream of one CUDA graph (the copy of
step s + 1 overlapping step s), each layer waiting for its own copy's event
and writing y straight into pinned host memory, PDL-chained on one
workspace, replayed several times."""
import numpy as np
import pytest
import torch

from flint_testlib import DeviceLayer, flint, margin_x
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 8])
def test_overlapped_host_copies_match_the_device_path(T):
    f = flint()
    k, H = 6, 1024
    layers = [DeviceLayer(synth.Layer(60 + i, H=H, E=16, I=256, I_shared=256)) for i in range(3)]
    xs = [margin_x(synth.bits(dl.L.router_w), T, H, k, None, seed=70 + i) for i, dl in enumerate(layers)]
    ws = layers[0].workspace(k)
    ids = [torch.empty((T, k), dtype=torch.int32, device="cuda") for _ in layers]
    w = [torch.empty((T, k), dtype=torch.float32, device="cuda") for _ in layers]

    # the device path, one call at a time
    ref = []
    for dl, x, i_, w_ in zip(layers, xs, ids, w):
        y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        f.flint_moe_layer(x.cuda(), dl.router_w, k, dl.routed, dl.shared, i_, w_, y, ws)
        torch.cuda.synchronize()
        ref.append(synth.bits(y))
    assert f.flint_workspace_check(ws) == f.FLINT_OK

    # the overlapped host-buffer graph: R steps cycling through the layers
    hx = [x.pin_memory() for x in xs]
    hy = [torch.zeros((T, H), dtype=torch.bfloat16).pin_memory() for _ in layers]
    dx = [torch.empty((T, H), dtype=torch.bfloat16, device="cuda") for _ in layers]
    R = 6
    stream, side = torch.cuda.Stream(), torch.cuda.Stream()

    def body():
        fork = torch.cuda.Event()
        fork.record(stream)
        side.wait_event(fork)
        evs = []
        with torch.cuda.stream(side):
            for s in range(R):
                dx[s % 3].copy_(hx[s % 3], non_blocking=True)
                e = torch.cuda.Event()
                e.record(side)
                evs.append(e)
        for s in range(R):
            li = s % 3
            stream.wait_event(evs[s])
            dl = layers[li]
            f.flint_moe_layer(dx[li], dl.router_w, k, dl.routed, dl.shared, ids[li], w[li], hy[li], ws,
                              flags=f.FLINT_PDL)

    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        for _ in range(3):
            g.replay()
        stream.synchronize()
    torch.cuda.synchronize()
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    for li in range(3):
        assert np.array_equal(synth.bits(hy[li]), ref[li]), f"layer {li}"
