"""CPU oracle for the Flint-style NVFP4 MoE decode step -- TEST INFRASTRUCTURE.

A ctypes front end over ``libflint_oracle.so`` (plain C, FP32 accumulation,
bf16 rounding at the method's stated points; see ``flint_oracle.c`` for the
definitions it follows and the readings it takes). Only the test suite, the
smoke check and the CPU-baseline leg of the benchmark may use it; the product
path never imports it.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None
_lib_omp = None
_active = None  # the library the functions below call (the plain build unless use_openmp)

W_NVFP4 = 0
W_BF16 = 1
EPI_NONE = 0
EPI_SWIGLU = 1


def _setup(L):
    L.fo_e2m1_value.restype = C.c_double
    L.fo_e2m1_value.argtypes = [C.c_int]
    L.fo_ue4m3_value.restype = C.c_double
    L.fo_ue4m3_value.argtypes = [C.c_int]
    L.fo_bf16_value.restype = C.c_double
    L.fo_bf16_value.argtypes = [C.c_uint16]
    L.fo_bf16_round.restype = C.c_uint16
    L.fo_bf16_round.argtypes = [C.c_double]
    L.fo_gguf_matrix_bytes.restype = C.c_int64
    L.fo_gguf_matrix_bytes.argtypes = [C.c_int64, C.c_int64]
    L.fo_packed_row_stride.restype = C.c_int64
    L.fo_packed_row_stride.argtypes = [C.c_int64]
    for name in ("fo_gguf_decode", "fo_packed_decode"):
        f = getattr(L, name)
        f.restype = C.c_int
        f.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p]
    L.fo_repack.restype = C.c_int
    L.fo_repack.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_int64, C.c_void_p, C.c_int64]
    L.fo_unrepack.restype = C.c_int
    L.fo_unrepack.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_int64, C.c_int64, C.c_void_p]
    L.fo_router.restype = C.c_int
    L.fo_router.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_int,
                            C.c_void_p, C.c_void_p, C.c_void_p]
    L.fo_expert.restype = C.c_int
    L.fo_expert.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p,
                            C.c_double, C.c_double, C.c_double, C.c_void_p, C.c_void_p, C.c_void_p,
                            C.c_void_p]
    L.fo_moe_experts.restype = C.c_int
    L.fo_moe_experts.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                 C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                 C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    L.fo_moe_layer.restype = C.c_int
    L.fo_moe_layer.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_int,
                               C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                               C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                               C.c_void_p, C.c_void_p, C.c_void_p]
    L.fo_dense_gemv.restype = C.c_int
    L.fo_dense_gemv.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_int, C.c_void_p,
                                C.c_int, C.c_void_p]
    L.fo_residual_rmsnorm.restype = C.c_int
    L.fo_residual_rmsnorm.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_double,
                                      C.c_void_p, C.c_void_p]
    L.fo_set_threads.restype = C.c_int
    L.fo_set_threads.argtypes = [C.c_int]
    return L


def lib():
    global _lib, _active
    if _lib is None:
        _lib = _setup(C.CDLL(_build.build()))
    if _active is None:
        _active = _lib
    return _active


def use_openmp(threads: int = 0) -> int:
    """Route the calls below to the OpenMP build with `threads` threads (0:
    all host threads); returns the thread count, or 0 (and keeps the plain
    build) where no OpenMP build exists. use_openmp(-1) returns to the plain
    build. Results are the same bits either way."""
    global _lib_omp, _active
    lib()
    if threads < 0:
        _active = _lib
        return 1
    if _lib_omp is None:
        path = _build.build_omp()
        if path is None:
            return 0
        _lib_omp = _setup(C.CDLL(path))
    _active = _lib_omp
    return _lib_omp.fo_set_threads(threads if threads > 0 else (os.cpu_count() or 1))


def _p(a):
    """Pointer of a C-contiguous numpy array, or None."""
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


# ---- formats --------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().fo_e2m1_value(code)


def ue4m3_value(byte: int) -> float:
    return lib().fo_ue4m3_value(byte)


def bf16_value(bits) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    f = np.vectorize(lib().fo_bf16_value, otypes=[np.float64])
    return f(bits) if bits.size else bits.astype(np.float64)


def bf16_round(values) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float64)
    f = np.vectorize(lib().fo_bf16_round, otypes=[np.uint16])
    return f(v) if v.size else v.astype(np.uint16)


def gguf_matrix_bytes(rows: int, cols: int) -> int:
    return lib().fo_gguf_matrix_bytes(rows, cols)


def packed_row_stride(cols: int) -> int:
    return lib().fo_packed_row_stride(cols)


def gguf_decode(src: np.ndarray, rows: int, cols: int) -> np.ndarray:
    out = np.empty((rows, cols), np.float64)
    _check(lib().fo_gguf_decode(_p(np.ascontiguousarray(src, np.uint8)), rows, cols, _p(out)), "gguf_decode")
    return out


def packed_decode(p: np.ndarray, rows: int, cols: int) -> np.ndarray:
    out = np.empty((rows, cols), np.float64)
    _check(lib().fo_packed_decode(_p(np.ascontiguousarray(p, np.uint8)), rows, cols, _p(out)), "packed_decode")
    return out


def repack(src: np.ndarray, n_mats: int, rows: int, cols: int, dst_mat_stride: int = 0) -> np.ndarray:
    ms = dst_mat_stride or rows * packed_row_stride(cols)
    dst = np.zeros(n_mats * ms, np.uint8)
    _check(lib().fo_repack(_p(np.ascontiguousarray(src, np.uint8)), n_mats, rows, cols, _p(dst), ms), "repack")
    return dst


def unrepack(dst: np.ndarray, n_mats: int, rows: int, cols: int, dst_mat_stride: int = 0) -> np.ndarray:
    src = np.zeros(n_mats * gguf_matrix_bytes(rows, cols), np.uint8)
    _check(lib().fo_unrepack(_p(np.ascontiguousarray(dst, np.uint8)), n_mats, rows, cols, dst_mat_stride,
                             _p(src)), "unrepack")
    return src


# ---- router / experts / layer ---------------------------------------------

def router(x, wr, k, bias=None):
    """x: uint16 bf16 bits [T, H]; wr: uint16 [E, H]; bias: float32 [E] or None.
    Returns (ids int32 [T,k], weights float64 [T,k], scores float32 [T,E])."""
    x = np.ascontiguousarray(x, np.uint16)
    wr = np.ascontiguousarray(wr, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    s = np.zeros((T, E), np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, np.float32)
    _check(lib().fo_router(_p(x), T, H, _p(wr), E, _p(b), k, _p(ids), _p(w), _p(s)), "router")
    return ids, w, s


def expert(x, gate, up, down, H, I, ts=(1.0, 1.0, 1.0), wdtype=W_NVFP4):
    """One token through one SwiGLU expert. Returns (g, u, h, d) as bf16 bits."""
    x = np.ascontiguousarray(x, np.uint16)
    g = np.zeros(I, np.uint16)
    u = np.zeros(I, np.uint16)
    h = np.zeros(I, np.uint16)
    d = np.zeros(H, np.uint16)
    _check(lib().fo_expert(_p(x), H, I, wdtype, _p(np.ascontiguousarray(gate)), _p(np.ascontiguousarray(up)),
                           _p(np.ascontiguousarray(down)), float(ts[0]), float(ts[1]), float(ts[2]),
                           _p(g), _p(u), _p(h), _p(d)), "expert")
    return g, u, h, d


def _opt(a, dtype=None):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype) if dtype is not None else np.ascontiguousarray(a)


def moe_experts(x, ids, weights, E, I, gate, up, down, ts=None, shared=None, wdtype=W_NVFP4):
    """Expert part of the layer given the routing. shared = None or a dict with
    keys gate, up, down, ts (3 floats), I."""
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    ids = np.ascontiguousarray(ids, np.int32)
    w = np.ascontiguousarray(weights, np.float32)
    k = ids.shape[1]
    y = np.zeros((T, H), np.uint16)
    sh = shared or {}
    keep = [_opt(gate), _opt(up), _opt(down), _opt(ts, np.float32), _opt(sh.get("gate")), _opt(sh.get("up")),
            _opt(sh.get("down")), _opt(sh.get("ts"), np.float32)]
    _check(lib().fo_moe_experts(_p(x), T, H, _p(ids), _p(w), k, E, I, wdtype, _p(keep[0]), _p(keep[1]),
                                _p(keep[2]), _p(keep[3]), int(sh.get("I", 0)), _p(keep[4]), _p(keep[5]),
                                _p(keep[6]), _p(keep[7]), _p(y)), "moe_experts")
    return y


def moe_layer(x, wr, k, E, I, gate, up, down, ts=None, shared=None, bias=None, wdtype=W_NVFP4):
    """Router + experts. Returns (ids, weights float32, y bf16 bits)."""
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    y = np.zeros((T, H), np.uint16)
    sh = shared or {}
    keep = [_opt(wr, np.uint16), _opt(bias, np.float32), _opt(gate), _opt(up), _opt(down), _opt(ts, np.float32),
            _opt(sh.get("gate")), _opt(sh.get("up")), _opt(sh.get("down")), _opt(sh.get("ts"), np.float32)]
    _check(lib().fo_moe_layer(_p(x), T, H, _p(keep[0]), E, _p(keep[1]), k, I, wdtype, _p(keep[2]), _p(keep[3]),
                              _p(keep[4]), _p(keep[5]), int(sh.get("I", 0)), _p(keep[6]), _p(keep[7]),
                              _p(keep[8]), _p(keep[9]), _p(ids), _p(w), _p(y)), "moe_layer")
    return ids, w, y


def dense_gemv(x, W, N, ts=(1.0, 1.0), epilogue=EPI_NONE, wdtype=W_NVFP4):
    x = np.ascontiguousarray(x, np.uint16)
    T, K = x.shape
    n_out = N // 2 if epilogue == EPI_SWIGLU else N
    y = np.zeros((T, n_out), np.uint16)
    tsa = np.ascontiguousarray(np.asarray(ts, np.float32))
    _check(lib().fo_dense_gemv(_p(x), T, K, wdtype, _p(np.ascontiguousarray(W)), N, _p(tsa), epilogue, _p(y)),
           "dense_gemv")
    return y


# ---- the decode stack: residual add + RMSNorm between blocks ----------------

def residual_rmsnorm(r, y=None, gamma=None, eps=1e-6):
    """r, y: uint16 bf16 bits [T, H] (y may be None); gamma: uint16 [H] or None.
    Returns (r' = bf16(r + y), x = bf16(rmsnorm(r') * gamma)) as bf16 bits."""
    r = np.ascontiguousarray(r, np.uint16)
    T, H = r.shape
    yy = None if y is None else np.ascontiguousarray(y, np.uint16)
    g = None if gamma is None else np.ascontiguousarray(gamma, np.uint16)
    r_out = np.zeros((T, H), np.uint16)
    x_out = np.zeros((T, H), np.uint16)
    _check(lib().fo_residual_rmsnorm(_p(r), _p(yy), T, H, _p(g), float(eps), _p(r_out), _p(x_out)),
           "residual_rmsnorm")
    return r_out, x_out


def decode_stack(x0, blocks, eps=1e-6):
    """One decode step of a pre-norm stack of MLP blocks (the attention of the
    model is outside this path): r = x0; for each block: r, x = norm(r + y),
    y = block(x); finally r = bf16(r + y). `blocks` holds dicts with kind
    "dense" (keys gate_up: GGUF bytes of the [2F, H] SwiGLU matrix, ts_gu: 2
    floats, down: GGUF bytes of [H, F], ts_down: 1 float, F) or kind "moe"
    (the keyword arguments of moe_layer plus wr and k). Returns (r_final, per
    block (x, y) bf16 bits, per MoE block ids)."""
    r = np.ascontiguousarray(x0, np.uint16)
    y = None
    trace, ids_all = [], []
    for b in blocks:
        r, x = residual_rmsnorm(r, y, None, eps)
        if b["kind"] == "dense":
            h = dense_gemv(x, b["gate_up"], 2 * b["F"], ts=b["ts_gu"], epilogue=EPI_SWIGLU)
            y = dense_gemv(h, b["down"], x.shape[1], ts=b["ts_down"], epilogue=EPI_NONE)
        else:
            args = {k: v for k, v in b.items() if k not in ("kind", "wr", "k")}
            ids, _, y = moe_layer(x, b["wr"], b["k"], **args)
            ids_all.append(ids)
        trace.append((x, y))
    r, _ = residual_rmsnorm(r, y, None, eps)
    return r, trace, ids_all
