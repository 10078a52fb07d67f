"""The C-ABI library loads, exports every function include/flint.h declares,
and rejects bad arguments on the host before touching a GPU (CPU only)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flint.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flint_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def flint():
    from nvfp4_moe_decode_sigmoid_gb300 import _build
    _build.build()
    from nvfp4_moe_decode_sigmoid_gb300 import flint as f
    return f


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("flint_nvfp4_repack", "flint_moe_route", "flint_moe_decode", "flint_dense_gemv",
              "flint_workspace_bytes", "flint_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(flint):
    lib = C.CDLL(flint.LIBRARY_PATH)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_size_helpers(flint):
    assert flint.flint_nvfp4_row_stride(2048) == 1152
    assert flint.flint_nvfp4_row_stride(512) == 288
    assert flint.flint_nvfp4_row_stride(64) == 48
    assert flint.flint_nvfp4_packed_bytes(256, 1024, 2048) == 256 * 1024 * 1152
    assert flint.flint_gguf_nvfp4_bytes(1, 2048, 512) == 2048 * 8 * 36
    ws = flint.flint_workspace_bytes(256, 6, 2048, 512, 512)
    # header, logits, h (routed, shared), d (routed, shared), row-block counters, per-expert counters
    need = (256 + 8 * 256 * 4 + 2 * 8 * 6 * 512 + 2 * 8 * 512 + 2 * 8 * 6 * 2048 + 2 * 8 * 2048 + 4 * 2048 // 16
            + 4 * (8 * 8 + 1))
    assert ws % 256 == 0 and ws >= need
    assert flint.flint_status_string(4) == "device wait timed out"


def _raw(flint):
    return flint.raw_library()


def test_host_validation_without_a_gpu(flint):
    L = _raw(flint)
    p = C.c_void_p(0x1000)  # aligned, never dereferenced: validation fails first
    # repack: cols not a multiple of 64
    assert L.flint_nvfp4_repack(p, 1, 4, 63, p, 0, None) == flint.FLINT_ERR_INVALID_ARG
    assert "cols" in flint.flint_last_error()
    # repack: stride too small
    assert L.flint_nvfp4_repack(p, 2, 4, 64, p, 16, None) == flint.FLINT_ERR_INVALID_ARG
    # route: batch outside 1..8, null pointers, bad k
    assert L.flint_moe_route(p, 9, 2048, p, 256, None, 6, p, p, p, 1 << 20, 0, None) == flint.FLINT_ERR_UNSUPPORTED
    assert L.flint_moe_route(None, 1, 2048, p, 256, None, 6, p, p, p, 1 << 20, 0, None) == flint.FLINT_ERR_INVALID_ARG
    assert L.flint_moe_route(p, 1, 2048, p, 256, None, 9, p, p, p, 1 << 20, 0, None) == flint.FLINT_ERR_UNSUPPORTED
    # route: misaligned x, small workspace
    assert L.flint_moe_route(C.c_void_p(0x1002), 1, 2048, p, 256, None, 6, p, p, p, 1 << 20, 0, None) == \
        flint.FLINT_ERR_INVALID_ARG
    assert L.flint_moe_route(p, 1, 2048, p, 256, None, 6, p, p, p, 64, 0, None) == flint.FLINT_ERR_INVALID_ARG
    # decode: missing routed experts, bad hidden size
    ex = flint.flint_experts(0, 256, 2048, 512, 0x1000, 0x1000, 0x1000)
    assert L.flint_moe_decode(p, 1, p, p, 6, None, None, p, p, 1 << 24, 0, None) == flint.FLINT_ERR_INVALID_ARG
    bad = flint.flint_experts(0, 256, 2000, 512, 0x1000, 0x1000, 0x1000)
    assert L.flint_moe_decode(p, 1, p, p, 6, C.byref(bad), None, p, p, 1 << 24, 0, None) == \
        flint.FLINT_ERR_UNSUPPORTED
    unk = flint.flint_experts(7, 256, 2048, 512, 0x1000, 0x1000, 0x1000)
    assert L.flint_moe_decode(p, 1, p, p, 6, C.byref(unk), None, p, p, 1 << 24, 0, None) == \
        flint.FLINT_ERR_UNSUPPORTED
    # BF16 experts: routed and shared must share the dtype; the one-kernel layer is NVFP4-only
    bf = flint.flint_experts(1, 256, 2048, 512, 0x1000, 0x1000, None)
    bf_sh = flint.flint_experts(0, 1, 2048, 512, 0x1000, 0x1000, 0x1000)
    assert L.flint_moe_decode(p, 1, p, p, 6, C.byref(bf), C.byref(bf_sh), p, p, 1 << 24, 0, None) == \
        flint.FLINT_ERR_UNSUPPORTED
    assert "same dtype" in flint.flint_last_error()
    assert L.flint_moe_layer(p, 1, p, 256, None, 6, C.byref(bf), None, p, p, p, p, 1 << 24, None, 0, None) == \
        flint.FLINT_ERR_UNSUPPORTED
    assert "NVFP4" in flint.flint_last_error()
    # the next layer's L2 prefetch ranges: 16-byte start and size, under 4 GiB in all
    ex4 = flint.flint_experts(0, 256, 2048, 512, 0x1000, 0x1000, 0x1000)
    for ptr, n in ((0x1008, 4096), (0x1000, 100), (0x1000, 1 << 32)):
        pf = flint.flint_l2_prefetch()
        pf.ptr[1], pf.bytes[1] = ptr, n
        assert L.flint_moe_layer(p, 1, p, 256, None, 6, C.byref(ex4), None, p, p, p, p, 1 << 24, C.byref(pf), 0,
                                 None) == flint.FLINT_ERR_INVALID_ARG
        assert "prefetch" in flint.flint_last_error()
    # NVFP4 experts need their tensor scales
    nots = flint.flint_experts(0, 256, 2048, 512, 0x1000, 0x1000, None)
    assert L.flint_moe_decode(p, 1, p, p, 6, C.byref(nots), None, p, p, 1 << 24, 0, None) == \
        flint.FLINT_ERR_INVALID_ARG
    sh = flint.flint_experts(0, 2, 2048, 512, 0x1000, 0x1000, 0x1000)
    assert L.flint_moe_decode(p, 1, p, p, 6, C.byref(ex), C.byref(sh), p, p, 1 << 24, 0, None) == \
        flint.FLINT_ERR_INVALID_ARG
    # decode: workspace too small
    assert L.flint_moe_gate_up(p, 1, p, 6, C.byref(ex), None, p, 1024, 0, None) == flint.FLINT_ERR_INVALID_ARG
    # dense: odd N with SwiGLU, K not a multiple of 256
    W = flint.flint_packed(0, 7, 2048, 0, 0x1000, 0x1000)
    assert L.flint_dense_gemv(p, 1, C.byref(W), 1, p, None, 0, 0, None) == flint.FLINT_ERR_UNSUPPORTED
    W2 = flint.flint_packed(0, 8, 512, 0, 0x1000, 0x1000)
    assert L.flint_dense_gemv(p, 1, C.byref(W2), 0, p, None, 0, 0, None) == flint.FLINT_ERR_UNSUPPORTED


def test_norm_validation_without_a_gpu(flint):
    L = _raw(flint)
    p = C.c_void_p(0x10000)
    q = C.c_void_p(0x20000)
    o = C.c_void_p(0x30000)
    n = flint.flint_norm(0x10000, None, None, 1e-6, 0.0, 0x20000, 0x30000)
    # x_out required for the standalone norm; H must be a multiple of 256
    nx = flint.flint_norm(0x10000, None, None, 1e-6, 0.0, 0x20000, None)
    assert L.flint_residual_rmsnorm(C.byref(nx), 1, 2048, 0, None) == flint.FLINT_ERR_INVALID_ARG
    assert L.flint_residual_rmsnorm(C.byref(n), 1, 2000, 0, None) == flint.FLINT_ERR_UNSUPPORTED
    assert L.flint_residual_rmsnorm(C.byref(n), 9, 2048, 0, None) == flint.FLINT_ERR_UNSUPPORTED
    assert L.flint_residual_rmsnorm(None, 1, 2048, 0, None) == flint.FLINT_ERR_INVALID_ARG
    # residual_out may not overlap the residual it is computed from
    ov = flint.flint_norm(0x10000, None, None, 1e-6, 0.0, 0x10400, 0x30000)
    assert L.flint_residual_rmsnorm(C.byref(ov), 1, 2048, 0, None) == flint.FLINT_ERR_INVALID_ARG
    assert "overlaps" in flint.flint_last_error()
    neg = flint.flint_norm(0x10000, None, None, -1.0, 0.0, 0x20000, 0x30000)
    assert L.flint_residual_rmsnorm(C.byref(neg), 1, 2048, 0, None) == flint.FLINT_ERR_INVALID_ARG
    # block: y may not overlap the norm's buffers
    ex = flint.flint_experts(0, 256, 2048, 512, 0x1000, 0x1000, 0x1000)
    assert L.flint_moe_block(C.byref(n), 1, p, 256, None, 6, C.byref(ex), None, p, p, C.c_void_p(0x20000), p,
                             1 << 24, None, 0, None) == flint.FLINT_ERR_INVALID_ARG
    assert L.flint_moe_block(None, 1, p, 256, None, 6, C.byref(ex), None, p, p, o, p, 1 << 24, None, 0, None) == \
        flint.FLINT_ERR_INVALID_ARG
    del q


@pytest.mark.parametrize("T,E", [(1, 1025), (4, 2048), (8, 1025)])
def test_static_router_rejects_more_experts_than_the_selection_keeps(flint, T, E):
    """flint_moe_route_static keeps at most 1024 scores per token, like
    flint_moe_route, even where its scratch would hold more (T = 1): larger E
    is rejected on the host."""
    L = _raw(flint)
    p = C.c_void_p(0x1000)
    st = L.flint_moe_route_static(p, T, 2048, p, E, None, 6, p, p, 0, None)
    assert st == flint.FLINT_ERR_UNSUPPORTED
    assert "limit of 1024" in flint.flint_last_error()
