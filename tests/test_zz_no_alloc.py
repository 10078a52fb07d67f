"""The router entry point for callers that cannot give the library device
memory (flint_moe_route_static, scratch inside the library) returns what the
workspace router (flint_moe_route) returns.

It is collected last, so a run that stops at its first failure has run every
other test before it. It passes on its own in a fresh process too.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from flint_testlib import flint, margin_x
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu


def _static_route(lib, x, wr, k, ids, w, bias, stream):
    f = lib.flint_moe_route_static
    f.restype = C.c_int
    f.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p,
                  C.c_uint, C.c_void_p]
    T, H = x.shape
    E = wr.shape[0]
    return f(C.c_void_p(x.data_ptr()), T, H, C.c_void_p(wr.data_ptr()), E,
             None if bias is None else C.c_void_p(bias.data_ptr()), k, C.c_void_p(ids.data_ptr()),
             C.c_void_p(w.data_ptr()), 0, C.c_void_p(stream.cuda_stream))


def test_static_scratch_router_matches_workspace_router_twice():
    F = flint()
    lib = F.raw_library()
    stream = torch.cuda.current_stream()
    # two calls in a row with different shapes: the second must not see
    # anything the first left in the shared scratch
    cases = [(256, 6, 2048, 8, None), (100, 4, 512, 3, synth.zipf_bias(2, 100))]
    for i, (E, k, H, T, bias) in enumerate(cases):
        wr = synth.bf16_normal(40 + i, (E, H), 0.02).cuda()
        x = margin_x(synth.bits(wr.cpu()), T, H, k, None if bias is None else bias.numpy(), seed=70 + i).cuda()
        b = None if bias is None else bias.cuda()
        ref_ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        ref_w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        ws = torch.empty(F.flint_workspace_bytes(E, k, 0, 0, 0), dtype=torch.uint8, device="cuda")
        F.flint_workspace_init(ws)
        F.flint_moe_route(x, wr, k, ref_ids, ref_w, ws, bias=b)
        ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        assert _static_route(lib, x, wr, k, ids, w, b, stream) == F.FLINT_OK, F.flint_last_error()
        torch.cuda.synchronize()
        a_ids, a_w = ids.cpu().numpy(), w.cpu().numpy()
        r_ids, r_w = ref_ids.cpu().numpy(), ref_w.cpu().numpy()
        for t in range(T):
            assert set(a_ids[t]) == set(r_ids[t])
            got = dict(zip(a_ids[t], a_w[t]))
            for e, we in zip(r_ids[t], r_w[t]):
                assert abs(got[e] - we) <= 2e-6 * we + 1e-7
        assert np.array_equal(a_ids, r_ids)


@pytest.mark.parametrize("T,E,why", [
    (8, 1025, "limit of 1024"),   # beyond both the selection and the 33,024-byte scratch
    (1, 1025, "limit of 1024"),   # fits the scratch, but the selection keeps 1024 scores per token
    (4, 2048, "limit of 1024"),
    (8, 1024, None),              # the largest accepted shape is not rejected by the size checks
])
def test_static_scratch_router_rejects_shapes_beyond_its_limits(T, E, why):
    F = flint()
    lib = F.raw_library()
    f = lib.flint_moe_route_static
    f.restype = C.c_int
    f.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p,
                  C.c_uint, C.c_void_p]
    if why is None:
        # a valid call: its inputs are real buffers of the right sizes
        H, k = 256, 6
        wr = synth.bf16_normal(90, (E, H), 0.02).cuda()
        x = synth.activations(91, T, H).cuda()
        ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        assert _static_route(lib, x, wr, k, ids, w, None, torch.cuda.current_stream()) == F.FLINT_OK
        torch.cuda.synchronize()
        assert bool((ids >= 0).all()) and bool((ids < E).all())
        return
    p = torch.empty(16, dtype=torch.int32, device="cuda")
    ptr = C.c_void_p(p.data_ptr())
    st = f(ptr, T, 2048, ptr, E, None, 6, ptr, ptr, 0, None)
    assert st == F.FLINT_ERR_UNSUPPORTED
    assert why in F.flint_last_error()
