"""Thin Python binding of libflint.so (the C ABI of include/flint.h).

Argument marshalling only: every function takes torch tensors (device memory
for the arrays), passes their pointers and sizes to the function of the same
name in the C library, and raises FlintError on a non-OK status. The current
torch CUDA stream is used unless a stream is given. The library must have
been built (``__graft_entry__.build()`` or ``python -m
nvfp4_moe_decode_sigmoid_gb300._build``); importing this module without it
fails loudly -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import _build

# FLINT_LIBRARY selects another build of the same C ABI (the phase-trace
# build of phase_trace.py); unset, the library built in this package.
_LIB_PATH = os.environ.get("FLINT_LIBRARY") or _build.LIB

FLINT_OK = 0
FLINT_ERR_INVALID_ARG = 1
FLINT_ERR_UNSUPPORTED = 2
FLINT_ERR_CUDA = 3
FLINT_ERR_TIMEOUT = 4

FLINT_DTYPE_NVFP4 = 0
FLINT_DTYPE_BF16 = 1
FLINT_EPILOGUE_NONE = 0
FLINT_EPILOGUE_SWIGLU = 1
FLINT_PDL = 1
FLINT_PDL_AFTER_ROUTE = 2
FLINT_MAX_TOKENS = 8


class FlintError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str):
        super().__init__(f"{what}: {detail} (status {status})")
        self.status = status


class flint_experts(C.Structure):
    _fields_ = [("dtype", C.c_int32), ("num_experts", C.c_int32), ("hidden", C.c_int32), ("inter", C.c_int32),
                ("gate_up", C.c_void_p), ("down", C.c_void_p), ("tensor_scale", C.c_void_p)]


class flint_packed(C.Structure):
    _fields_ = [("dtype", C.c_int32), ("rows", C.c_int32), ("cols", C.c_int32), ("reserved", C.c_int32),
                ("data", C.c_void_p), ("tensor_scale", C.c_void_p)]


class flint_norm(C.Structure):
    _fields_ = [("residual", C.c_void_p), ("y", C.c_void_p), ("gamma", C.c_void_p), ("eps", C.c_float),
                ("reserved", C.c_float), ("residual_out", C.c_void_p), ("x_out", C.c_void_p)]


class flint_l2_prefetch(C.Structure):
    _fields_ = [("ptr", C.c_void_p * 4), ("bytes", C.c_size_t * 4)]


def l2_prefetch(*tensors):
    """The next layer's weights (up to four device tensors, each 16-byte
    aligned with a size that is a multiple of 16) for flint_moe_layer /
    flint_moe_block to pull into L2 before their PDL wait."""
    assert len(tensors) <= 4
    p = flint_l2_prefetch()
    for i, t in enumerate(tensors):
        p.ptr[i] = t.data_ptr()
        p.bytes[i] = t.numel() * t.element_size()
    return p


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libflint.so is not built ({_LIB_PATH}); run __graft_entry__.build() first")
    L = C.CDLL(_LIB_PATH)
    vp, i32, i64, u32, sz = C.c_void_p, C.c_int, C.c_int64, C.c_uint, C.c_size_t
    sig = {
        "flint_last_error": (C.c_char_p, []),
        "flint_status_string": (C.c_char_p, [i32]),
        "flint_nvfp4_row_stride": (i64, [i64]),
        "flint_nvfp4_packed_bytes": (i64, [i64, i64, i64]),
        "flint_gguf_nvfp4_bytes": (i64, [i64, i64, i64]),
        "flint_workspace_bytes": (sz, [i32, i32, i32, i32, i32]),
        "flint_workspace_set_wait_budget": (i32, [vp, sz, u32, vp]),
        "flint_selftest_lose_cta": (i32, [vp, sz, i32, vp]),
        "flint_workspace_init": (i32, [vp, sz, vp]),
        "flint_workspace_check": (i32, [vp, sz, vp]),
        "flint_nvfp4_repack": (i32, [vp, i64, i64, i64, vp, i64, vp]),
        "flint_nvfp4_unrepack": (i32, [vp, i64, i64, i64, i64, vp, vp]),
        "flint_nvfp4_dequant": (i32, [vp, i64, i64, vp, vp]),
        "flint_moe_route": (i32, [vp, i32, i32, vp, i32, vp, i32, vp, vp, vp, sz, u32, vp]),
        "flint_moe_gate_up": (i32, [vp, i32, vp, i32, C.POINTER(flint_experts), C.POINTER(flint_experts), vp, sz,
                                    u32, vp]),
        "flint_moe_down_combine": (i32, [i32, vp, vp, i32, C.POINTER(flint_experts), C.POINTER(flint_experts), vp,
                                         vp, sz, u32, vp]),
        "flint_moe_decode": (i32, [vp, i32, vp, vp, i32, C.POINTER(flint_experts), C.POINTER(flint_experts), vp, vp,
                                   sz, u32, vp]),
        "flint_dense_gemv": (i32, [vp, i32, C.POINTER(flint_packed), i32, vp, vp, sz, u32, vp]),
        "flint_selftest_wait_timeout": (i32, [vp, sz, C.c_uint64, vp]),
        "flint_moe_route_static": (i32, [vp, i32, i32, vp, i32, vp, i32, vp, vp, u32, vp]),
        "flint_moe_layer": (i32, [vp, i32, vp, i32, vp, i32, C.POINTER(flint_experts), C.POINTER(flint_experts), vp,
                                  vp, vp, vp, sz, C.POINTER(flint_l2_prefetch), u32, vp]),
        "flint_residual_rmsnorm": (i32, [C.POINTER(flint_norm), i32, i32, u32, vp]),
        "flint_prefill_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32]),
        "flint_moe_prefill": (i32, [vp, i32, vp, i32, vp, i32, C.POINTER(flint_experts), C.POINTER(flint_experts),
                                    vp, vp, vp, vp, sz, u32, vp]),
        "flint_moe_block": (i32, [C.POINTER(flint_norm), i32, vp, i32, vp, i32, C.POINTER(flint_experts),
                                  C.POINTER(flint_experts), vp, vp, vp, vp, sz, C.POINTER(flint_l2_prefetch), u32,
                                  vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


_lib = _load()
LIBRARY_PATH = _LIB_PATH


def _ptr(t):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def _check(status: int, what: str):
    if status != FLINT_OK:
        raise FlintError(status, what, _lib.flint_last_error().decode())


# ---------------------------------------------------------------------------
# sizes
# ---------------------------------------------------------------------------
def flint_nvfp4_row_stride(cols: int) -> int:
    return _lib.flint_nvfp4_row_stride(cols)


def flint_nvfp4_packed_bytes(n_mats: int, rows: int, cols: int) -> int:
    return _lib.flint_nvfp4_packed_bytes(n_mats, rows, cols)


def flint_gguf_nvfp4_bytes(n_mats: int, rows: int, cols: int) -> int:
    return _lib.flint_gguf_nvfp4_bytes(n_mats, rows, cols)


def flint_workspace_bytes(num_experts: int, top_k: int, hidden: int, inter: int, inter_shared: int) -> int:
    return _lib.flint_workspace_bytes(num_experts, top_k, hidden, inter, inter_shared)


def flint_last_error() -> str:
    return _lib.flint_last_error().decode()


def flint_status_string(status: int) -> str:
    return _lib.flint_status_string(status).decode()


# ---------------------------------------------------------------------------
# workspace
# ---------------------------------------------------------------------------
def flint_workspace_init(ws: torch.Tensor, stream=None):
    _check(_lib.flint_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "workspace_init")


def flint_workspace_check(ws: torch.Tensor, stream=None) -> int:
    """Returns the status (FLINT_OK or FLINT_ERR_TIMEOUT / INVALID_ARG) without raising."""
    return _lib.flint_workspace_check(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


# ---------------------------------------------------------------------------
# packing
# ---------------------------------------------------------------------------
def flint_nvfp4_repack(src: torch.Tensor, n_mats: int, rows: int, cols: int, dst: torch.Tensor,
                       dst_mat_stride: int = 0, dst_offset: int = 0, stream=None):
    dptr = C.c_void_p(dst.data_ptr() + dst_offset)
    _check(_lib.flint_nvfp4_repack(_ptr(src), n_mats, rows, cols, dptr, dst_mat_stride, _stream(stream)), "repack")


def flint_nvfp4_unrepack(dst: torch.Tensor, n_mats: int, rows: int, cols: int, src: torch.Tensor,
                         dst_mat_stride: int = 0, dst_offset: int = 0, stream=None):
    dptr = C.c_void_p(dst.data_ptr() + dst_offset)
    _check(_lib.flint_nvfp4_unrepack(dptr, n_mats, rows, cols, dst_mat_stride, _ptr(src), _stream(stream)),
           "unrepack")


def flint_nvfp4_dequant(packed: torch.Tensor, rows: int, cols: int, out: torch.Tensor, stream=None):
    _check(_lib.flint_nvfp4_dequant(_ptr(packed), rows, cols, _ptr(out), _stream(stream)), "dequant")


# ---------------------------------------------------------------------------
# experts
# ---------------------------------------------------------------------------
class Experts:
    """Device weights of E experts in the kernel layout plus their C descriptor.

    gate_up: uint8 [E * 2I * row_stride(H)], down: uint8 [E * H * row_stride(I)],
    tensor_scale: float32 [E, 3].
    """

    def __init__(self, gate_up, down, tensor_scale, num_experts, hidden, inter, dtype=FLINT_DTYPE_NVFP4):
        self.gate_up, self.down, self.tensor_scale = gate_up, down, tensor_scale
        self.num_experts, self.hidden, self.inter, self.dtype = num_experts, hidden, inter, dtype
        self.struct = flint_experts(dtype, num_experts, hidden, inter, gate_up.data_ptr(),
                                    down.data_ptr() if down is not None else None,
                                    tensor_scale.data_ptr() if tensor_scale is not None else None)

    @property
    def packed_bytes(self) -> int:
        return self.gate_up.numel() + (self.down.numel() if self.down is not None else 0)

    @staticmethod
    def from_gguf(gate, up, down, tensor_scale, num_experts, hidden, inter, stream=None):
        """Repack GGUF NVFP4 gate [E, I, H], up [E, I, H], down [E, H, I] (device
        uint8 tensors) into the kernel layout: gate rows [0, I) and up rows
        [I, 2I) of each expert's [2I, H] gate/up matrix."""
        dev = gate.device
        rs_h = flint_nvfp4_row_stride(hidden)
        gu = torch.empty(num_experts * 2 * inter * rs_h, dtype=torch.uint8, device=dev)
        dn = torch.empty(flint_nvfp4_packed_bytes(num_experts, hidden, inter), dtype=torch.uint8, device=dev)
        stride = 2 * inter * rs_h
        flint_nvfp4_repack(gate, num_experts, inter, hidden, gu, stride, 0, stream)
        flint_nvfp4_repack(up, num_experts, inter, hidden, gu, stride, inter * rs_h, stream)
        flint_nvfp4_repack(down, num_experts, hidden, inter, dn, 0, 0, stream)
        ts = tensor_scale.to(device=dev, dtype=torch.float32).contiguous()
        return Experts(gu, dn, ts, num_experts, hidden, inter)


    @staticmethod
    def from_bf16(gate, up, down, num_experts, hidden, inter, tensor_scale=None):
        """BF16 experts: gate [E, I, H], up [E, I, H], down [E, H, I] (device
        bf16 tensors) -> the [E, 2I, H] gate/up matrices (gate rows first) and
        down as given. tensor_scale: None (all 1) or float32 [E, 3]."""
        E, I, H = num_experts, inter, hidden
        gu = torch.cat([gate.reshape(E, I, H), up.reshape(E, I, H)], dim=1).contiguous()
        dn = down.reshape(E, H, I).contiguous()
        ts = tensor_scale.to(device=gu.device, dtype=torch.float32).contiguous() if tensor_scale is not None else None
        return Experts(gu, dn, ts, E, H, I, dtype=FLINT_DTYPE_BF16)


class Packed:
    """A dense [N, K] NVFP4 matrix in the kernel layout plus its C descriptor."""

    def __init__(self, data, rows, cols, tensor_scale, dtype=FLINT_DTYPE_NVFP4):
        self.data, self.rows, self.cols, self.tensor_scale = data, rows, cols, tensor_scale
        self.struct = flint_packed(dtype, rows, cols, 0, data.data_ptr(), tensor_scale.data_ptr())

    @staticmethod
    def from_gguf(src, rows, cols, tensor_scale, stream=None):
        dev = src.device
        d = torch.empty(flint_nvfp4_packed_bytes(1, rows, cols), dtype=torch.uint8, device=dev)
        flint_nvfp4_repack(src, 1, rows, cols, d, 0, 0, stream)
        return Packed(d, rows, cols, tensor_scale.to(device=dev, dtype=torch.float32).contiguous())


def _ex(e):
    return C.byref(e.struct) if e is not None else None


# ---------------------------------------------------------------------------
# MoE layer
# ---------------------------------------------------------------------------
def flint_moe_route(x, router_w, k, ids, weights, ws, bias=None, flags=0, stream=None):
    T, H = x.shape
    E = router_w.shape[0]
    _check(_lib.flint_moe_route(_ptr(x), T, H, _ptr(router_w), E, _ptr(bias), k, _ptr(ids), _ptr(weights), _ptr(ws),
                                ws.numel() * ws.element_size(), flags, _stream(stream)), "moe_route")


def flint_moe_gate_up(x, ids, routed: Experts, shared: Experts | None, ws, flags=0, stream=None):
    T = x.shape[0]
    k = ids.shape[1]
    _check(_lib.flint_moe_gate_up(_ptr(x), T, _ptr(ids), k, _ex(routed), _ex(shared), _ptr(ws),
                                  ws.numel() * ws.element_size(), flags, _stream(stream)), "moe_gate_up")


def flint_moe_down_combine(ids, weights, routed: Experts, shared: Experts | None, y, ws, flags=0, stream=None):
    T, k = ids.shape
    _check(_lib.flint_moe_down_combine(T, _ptr(ids), _ptr(weights), k, _ex(routed), _ex(shared), _ptr(y), _ptr(ws),
                                       ws.numel() * ws.element_size(), flags, _stream(stream)), "moe_down_combine")


def flint_moe_decode(x, ids, weights, routed: Experts, shared: Experts | None, y, ws, flags=0, stream=None):
    T = x.shape[0]
    k = ids.shape[1]
    _check(_lib.flint_moe_decode(_ptr(x), T, _ptr(ids), _ptr(weights), k, _ex(routed), _ex(shared), _ptr(y),
                                 _ptr(ws), ws.numel() * ws.element_size(), flags, _stream(stream)), "moe_decode")


def flint_moe_layer(x, router_w, k, routed: Experts, shared: Experts | None, ids, weights, y, ws, bias=None, flags=0,
                    stream=None, next=None):
    """The whole layer in one launch: routing (ids, weights written) and y.
    next: l2_prefetch(...) of the next layer's weights, or None."""
    T = x.shape[0]
    E = router_w.shape[0]
    _check(_lib.flint_moe_layer(_ptr(x), T, _ptr(router_w), E, _ptr(bias), k, _ex(routed), _ex(shared), _ptr(ids),
                                _ptr(weights), _ptr(y), _ptr(ws), ws.numel() * ws.element_size(),
                                C.byref(next) if next is not None else None, flags, _stream(stream)), "moe_layer")


def _norm(residual, y_prev, gamma, eps, residual_out, x_out):
    return flint_norm(residual.data_ptr(), y_prev.data_ptr() if y_prev is not None else None,
                      gamma.data_ptr() if gamma is not None else None, float(eps), 0.0,
                      residual_out.data_ptr() if residual_out is not None else None,
                      x_out.data_ptr() if x_out is not None else None)


def flint_residual_rmsnorm(residual, x_out, y_prev=None, residual_out=None, gamma=None, eps=1e-6, flags=0,
                           stream=None):
    """r' = bf16(residual + y_prev) into residual_out (when given) and
    x = bf16(rmsnorm(r') * gamma) into x_out; all [T, H] bf16 (gamma [H])."""
    T, H = residual.shape
    n = _norm(residual, y_prev, gamma, eps, residual_out, x_out)
    _check(_lib.flint_residual_rmsnorm(C.byref(n), T, H, flags, _stream(stream)), "residual_rmsnorm")


def flint_moe_block(residual, router_w, k, routed: Experts, shared: Experts | None, ids, weights, y, ws,
                    y_prev=None, residual_out=None, x_out=None, gamma=None, eps=1e-6, bias=None, flags=0,
                    stream=None, next=None):
    """One pre-norm MoE block in one launch: x = rmsnorm(residual + y_prev)
    (residual_out receives the sum), then the MoE layer on x into y.
    next: l2_prefetch(...) of the next block's weights, or None."""
    T = residual.shape[0]
    E = router_w.shape[0]
    n = _norm(residual, y_prev, gamma, eps, residual_out, x_out)
    _check(_lib.flint_moe_block(C.byref(n), T, _ptr(router_w), E, _ptr(bias), k, _ex(routed), _ex(shared),
                                _ptr(ids), _ptr(weights), _ptr(y), _ptr(ws), ws.numel() * ws.element_size(),
                                C.byref(next) if next is not None else None, flags, _stream(stream)), "moe_block")


def flint_prefill_workspace_bytes(tokens: int, num_experts: int, top_k: int, hidden: int, inter: int,
                                  inter_shared: int) -> int:
    return _lib.flint_prefill_workspace_bytes(tokens, num_experts, top_k, hidden, inter, inter_shared)


def flint_moe_prefill(x, router_w, k, routed: Experts, shared: Experts | None, ids, weights, y, ws, bias=None,
                      stream=None):
    """The MoE layer over T tokens on the tensor cores (router GEMM, top-k,
    expert sort, grouped gate/up and down GEMMs, combine)."""
    T = x.shape[0]
    E = router_w.shape[0]
    _check(_lib.flint_moe_prefill(_ptr(x), T, _ptr(router_w), E, _ptr(bias), k, _ex(routed), _ex(shared), _ptr(ids),
                                  _ptr(weights), _ptr(y), _ptr(ws), ws.numel() * ws.element_size(), 0,
                                  _stream(stream)), "moe_prefill")


def flint_dense_gemv(x, W: Packed, y, epilogue=FLINT_EPILOGUE_NONE, ws=None, flags=0, stream=None):
    T = x.shape[0]
    wsb = ws.numel() * ws.element_size() if ws is not None else 0
    _check(_lib.flint_dense_gemv(_ptr(x), T, C.byref(W.struct), epilogue, _ptr(y), _ptr(ws), wsb, flags,
                                 _stream(stream)), "dense_gemv")


def flint_moe_route_static(x, router_w, k, ids, weights, bias=None, flags=0, stream=None):
    """flint_moe_route for callers that cannot hand the library a workspace:
    the scratch is a fixed array inside the library (see include/flint.h)."""
    T, H = x.shape
    E = router_w.shape[0]
    _check(_lib.flint_moe_route_static(_ptr(x), T, H, _ptr(router_w), E, _ptr(bias), k, _ptr(ids), _ptr(weights),
                                       flags, _stream(stream)), "moe_route_static")


def flint_selftest_wait_timeout(ws, budget_ns: int, stream=None):
    _check(_lib.flint_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(), budget_ns, _stream(stream)),
           "selftest_wait_timeout")


def flint_workspace_set_wait_budget(ws, budget_us: int, stream=None):
    _check(_lib.flint_workspace_set_wait_budget(_ptr(ws), ws.numel() * ws.element_size(), budget_us,
                                                _stream(stream)), "workspace_set_wait_budget")


def flint_selftest_lose_cta(ws, cta: int, stream=None):
    _check(_lib.flint_selftest_lose_cta(_ptr(ws), ws.numel() * ws.element_size(), cta, _stream(stream)),
           "selftest_lose_cta")


def raw_library():
    """The ctypes handle, for callers that marshal their own arguments."""
    return _lib
