"""GPU residual add + RMSNorm (standalone and fused into the MoE block) and a
short pre-norm decode stack against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from flint_testlib import DeviceLayer, MARGIN, assert_close, bf16_to_f64, combine_terms, flint
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu

EPS = 1e-6


def within_one_ulp(gpu_bits, ref_bits):
    """bf16 values equal, or one unit in the last place of the reference apart
    (the FP32 norm and the oracle's double norm may round a value near a bf16
    rounding boundary differently)."""
    a, r = bf16_to_f64(gpu_bits), bf16_to_f64(ref_bits)
    mag = np.maximum(np.abs(r), 2.0 ** -126)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
    return np.abs(a - r) <= ulp * (1 + 1e-12)


def residual_pair(seed, T, H, y_scale=0.5):
    r = synth.activations(seed, T, H)
    y = (synth.activations(seed + 7919, T, H).float() * y_scale).to(torch.bfloat16)
    return r, y


@pytest.mark.parametrize("T,H,with_y,with_gamma", [(1, 2048, True, False), (3, 1024, False, False),
                                                   (8, 2048, True, True), (5, 4096, True, False),
                                                   (2, 256, True, True)])
def test_rmsnorm_standalone(T, H, with_y, with_gamma):
    f = flint()
    r, y = residual_pair(100 + T, T, H)
    gamma = synth.bf16_normal(55, (H,), 1.0) if with_gamma else None
    r_out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    x_out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    f.flint_residual_rmsnorm(r.cuda(), x_out, y_prev=y.cuda() if with_y else None, residual_out=r_out,
                             gamma=gamma.cuda() if with_gamma else None, eps=EPS)
    torch.cuda.synchronize()
    rr, rx = oracle.residual_rmsnorm(synth.bits(r), synth.bits(y) if with_y else None,
                                     synth.bits(gamma) if with_gamma else None, EPS)
    assert np.array_equal(synth.bits(r_out), rr)
    ok = within_one_ulp(synth.bits(x_out), rx)
    assert ok.all(), f"{int((~ok).sum())} values more than one ulp off"
    assert (synth.bits(x_out) == rx).mean() > 0.99


def test_rmsnorm_zero_residual_gives_zero():
    f = flint()
    r, _ = residual_pair(3, 2, 1024)
    neg = (-r.float()).to(torch.bfloat16)
    x_out = torch.full((2, 1024), 7.0, dtype=torch.bfloat16, device="cuda")
    f.flint_residual_rmsnorm(r.cuda(), x_out, y_prev=neg.cuda(), eps=EPS)
    torch.cuda.synchronize()
    assert torch.all(x_out == 0)


def block_inputs(router_bits, T, H, k, seed, margin=MARGIN):
    """Residual r and previous output y per token, resampled until the oracle's
    normalised x = rmsnorm(r + y) has a top-k score margin of at least `margin`."""
    rs, ys = [], []
    for t in range(T):
        rep = 0
        while True:
            r, y = residual_pair(seed * 1000003 + t * 10007 + rep, 1, H)
            _, x = oracle.residual_rmsnorm(synth.bits(r), synth.bits(y), None, EPS)
            _, _, s = oracle.router(x, router_bits, k)
            ss = np.sort(s[0])[::-1]
            if ss[k - 1] - ss[k] >= margin:
                break
            rep += 1
        rs.append(r)
        ys.append(y)
    return torch.cat(rs), torch.cat(ys)


def run_block(dl, r, y_prev, k, flags=0, bias=None):
    f = flint()
    T, H = r.shape
    ws = dl.workspace(k)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    r_out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    x_out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    f.flint_moe_block(r.cuda(), dl.router_w, k, dl.routed, dl.shared, ids, w, y, ws, y_prev=y_prev.cuda(),
                      residual_out=r_out, x_out=x_out, eps=EPS, bias=bias, flags=flags)
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    return [synth.bits(t) if t.dtype == torch.bfloat16 else t.cpu().numpy() for t in (ids, w, y, r_out, x_out)]


def check_block(dl, r, y_prev, k, flags=0):
    ids, w, y, r_out, x_out = run_block(dl, r, y_prev, k, flags)
    rr, rx = oracle.residual_rmsnorm(synth.bits(r), synth.bits(y_prev), None, EPS)
    assert np.array_equal(r_out, rr)
    assert within_one_ulp(x_out, rx).all()
    # routing from the oracle's own norm (the inputs keep the top-k margin)
    rids, rw, _ = oracle.moe_layer(rx, synth.bits(dl.L.router_w), k, **dl.oracle_args())
    for t in range(r.shape[0]):
        assert set(ids[t]) == set(rids[t])
    # the layer on the block's own normalised input (checked above against
    # the oracle's norm to one ulp): the same inputs on both sides
    gids, gw, gy = oracle.moe_layer(x_out, synth.bits(dl.L.router_w), k, **dl.oracle_args())
    assert np.array_equal(ids, gids)
    assert_close(y, gy, "block", terms=combine_terms(x_out, gids, gw, dl))
    return ids, y


@pytest.fixture(scope="module")
def small_layer():
    return DeviceLayer(synth.Layer(31, H=1024, E=16, I=256, I_shared=256))


@pytest.mark.parametrize("T,k", [(1, 6), (4, 2), (8, 6)])
def test_small_block(small_layer, T, k):
    r, y = block_inputs(synth.bits(small_layer.L.router_w), T, 1024, k, seed=T + 10 * k)
    check_block(small_layer, r, y, k)


def test_small_block_pdl_is_bitwise_identical(small_layer):
    f = flint()
    r, y = block_inputs(synth.bits(small_layer.L.router_w), 8, 1024, 6, seed=77)
    a = run_block(small_layer, r, y, 6, flags=0)
    b = run_block(small_layer, r, y, 6, flags=f.FLINT_PDL)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_block_norm_matches_standalone_norm(small_layer):
    """The fused norm and the standalone kernel sum in the same order: same bits."""
    f = flint()
    r, y = block_inputs(synth.bits(small_layer.L.router_w), 8, 1024, 6, seed=78)
    _, _, _, r_out, x_out = run_block(small_layer, r, y, 6)
    x2 = torch.empty((8, 1024), dtype=torch.bfloat16, device="cuda")
    r2 = torch.empty((8, 1024), dtype=torch.bfloat16, device="cuda")
    f.flint_residual_rmsnorm(r.cuda(), x2, y_prev=y.cuda(), residual_out=r2, eps=EPS)
    torch.cuda.synchronize()
    assert np.array_equal(synth.bits(x2), x_out) and np.array_equal(synth.bits(r2), r_out)


@pytest.fixture(scope="module")
def full_layer():
    return DeviceLayer(synth.Layer(1005))


@pytest.mark.parametrize("T", [1, 8])
def test_full_block(full_layer, T):
    f = flint()
    r, y = block_inputs(synth.bits(full_layer.L.router_w), T, 2048, 6, seed=300 + T)
    check_block(full_layer, r, y, 6, flags=f.FLINT_PDL)


# ---------------------------------------------------------------------------
# a short decode stack: dense block, then MoE blocks, residual + norm between
# ---------------------------------------------------------------------------
H_S, F_S, E_S, I_S = 1024, 2048, 32, 256


def stack_blocks(n_moe, seed):
    blocks = []
    gu = synth.gguf_nvfp4(seed * 7 + 1, 1, 2 * F_S, H_S)
    dn = synth.gguf_nvfp4(seed * 7 + 2, 1, H_S, F_S)
    ts = synth.tensor_scales(seed * 7 + 3, (3,))
    blocks.append(dict(kind="dense", F=F_S, gate_up=gu.numpy(), ts_gu=tuple(ts[:2].tolist()), down=dn.numpy(),
                       ts_down=(float(ts[2]),), _t=(gu, dn, ts)))
    for i in range(n_moe):
        L = synth.Layer(seed * 7 + 10 + i, H=H_S, E=E_S, I=I_S, I_shared=I_S)
        blocks.append(dict(kind="moe", _L=L))
    return blocks


def oracle_blocks(blocks, k):
    out = []
    for b in blocks:
        if b["kind"] == "dense":
            out.append({kk: v for kk, v in b.items() if not kk.startswith("_")})
        else:
            L = b["_L"]
            sh = L.shared
            out.append(dict(kind="moe", wr=synth.bits(L.router_w), k=k, E=L.E, I=L.I, gate=L.gate.numpy(),
                            up=L.up.numpy(), down=L.down.numpy(), ts=L.ts.numpy(),
                            shared=dict(gate=sh["gate"].numpy(), up=sh["up"].numpy(), down=sh["down"].numpy(),
                                        ts=sh["ts"].numpy(), I=sh["I"])))
    return out


def stack_x0(blocks, T, k, seed, margin=2 * MARGIN):
    """Seeded input tokens for which every MoE block of the oracle's stack has
    a top-k margin of at least `margin` (so both sides route alike)."""
    ob = oracle_blocks(blocks, k)
    rep = 0
    while True:
        x0 = synth.activations(seed * 131 + rep, T, H_S)
        _, trace, _ = oracle.decode_stack(synth.bits(x0), ob, EPS)
        ok = True
        for b, (x, _) in zip(ob, trace):
            if b["kind"] != "moe":
                continue
            _, _, s = oracle.router(x, b["wr"], k)
            ss = np.sort(s, axis=1)[:, ::-1]
            ok = ok and bool(np.all(ss[:, k - 1] - ss[:, k] >= margin))
        if ok:
            return x0, ob
        rep += 1


def run_stack(f, blocks, x0, k, flags, record=False):
    """The stack on the GPU through the C ABI: standalone norm + dense SwiGLU
    GEMV + dense GEMV for the dense block, one flint_moe_block per MoE block,
    a final standalone residual add. With `record`, also each block's inputs
    (residual, previous output), its normalised input x and its output, as
    bf16 bits."""
    T = x0.shape[0]
    dev = "cuda"
    rbuf = [x0.cuda().contiguous(), torch.empty((T, H_S), dtype=torch.bfloat16, device=dev)]
    ybuf = [torch.empty((T, H_S), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    x = torch.empty((T, H_S), dtype=torch.bfloat16, device=dev)
    h = torch.empty((T, F_S), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(f.flint_workspace_bytes(E_S, k, H_S, I_S, I_S), dtype=torch.uint8, device=dev)
    f.flint_workspace_init(ws)
    ids_all, seen = [], []
    cur, y_prev = 0, None
    for i, b in enumerate(blocks):
        y = ybuf[i % 2]
        r_in = rbuf[cur]
        y_in = y_prev
        if b["kind"] == "dense":
            if "_dev" not in b:
                gu, dn, ts = b["_t"]
                b["_dev"] = (f.Packed.from_gguf(gu.cuda(), 2 * F_S, H_S, ts[:2].cuda()),
                             f.Packed.from_gguf(dn.cuda(), H_S, F_S, ts[2:].cuda()))
            Wgu, Wdn = b["_dev"]
            f.flint_residual_rmsnorm(rbuf[cur], x, y_prev=y_prev, residual_out=rbuf[1 - cur] if y_prev is not None
                                     else None, eps=EPS, flags=flags)
            if y_prev is not None:
                cur = 1 - cur
            f.flint_dense_gemv(x, Wgu, h, epilogue=f.FLINT_EPILOGUE_SWIGLU, flags=flags)
            f.flint_dense_gemv(h, Wdn, y, epilogue=f.FLINT_EPILOGUE_NONE, flags=flags)
        else:
            if "_dl" not in b:
                b["_dl"] = DeviceLayer(b["_L"])
            dl = b["_dl"]
            ids = torch.empty((T, k), dtype=torch.int32, device=dev)
            w = torch.empty((T, k), dtype=torch.float32, device=dev)
            f.flint_moe_block(rbuf[cur], dl.router_w, k, dl.routed, dl.shared, ids, w, y, ws, y_prev=y_prev,
                              residual_out=rbuf[1 - cur], x_out=x if record else None, eps=EPS, flags=flags)
            cur = 1 - cur
            ids_all.append(ids)
        if record:
            torch.cuda.synchronize()
            seen.append(tuple(None if t is None else synth.bits(t) for t in (r_in, y_in, x, y)))
        y_prev = y
    r_final = torch.empty((T, H_S), dtype=torch.bfloat16, device=dev)
    xf = torch.empty((T, H_S), dtype=torch.bfloat16, device=dev)
    f.flint_residual_rmsnorm(rbuf[cur], xf, y_prev=y_prev, residual_out=r_final, eps=EPS, flags=flags)
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    if record:
        return synth.bits(r_final), [i.cpu().numpy() for i in ids_all], seen
    return synth.bits(r_final), [i.cpu().numpy() for i in ids_all]


@pytest.fixture(scope="module")
def stack():
    blocks = stack_blocks(3, seed=5)
    x0, ob = stack_x0(blocks, 2, 6, seed=5)
    return blocks, x0, ob


def test_short_stack_matches_oracle(stack):
    """Every block of the GPU's stack against the oracle's block on the same
    inputs: the GPU's norm of its residual stream and previous output to one
    ulp of the oracle's, and the block's output, from the GPU's normalised
    input, within the layer tolerance. The whole stack against the oracle's own stack: the same
    routing in every block, and the final residual within relative L2 1e-2
    (both sides round in FP32 in different orders at every block, and the
    per-element bound is for one layer, not for a chain of them)."""
    f = flint()
    blocks, x0, ob = stack
    k = 6
    r, ids, seen = run_stack(f, blocks, x0, k, flags=0, record=True)
    for blk, b, (r_in, y_in, x, y_out) in zip(blocks, ob, seen):
        _, rx = oracle.residual_rmsnorm(r_in, y_in, None, EPS)
        assert within_one_ulp(x, rx).all()
        if b["kind"] == "dense":
            hh = oracle.dense_gemv(x, b["gate_up"], 2 * b["F"], ts=b["ts_gu"], epilogue=oracle.EPI_SWIGLU)
            ry = oracle.dense_gemv(hh, b["down"], x.shape[1], ts=b["ts_down"], epilogue=oracle.EPI_NONE)
            assert_close(y_out, ry, "dense block")
        else:
            args = {kk: v for kk, v in b.items() if kk not in ("kind", "wr", "k")}
            gids, gw, gy = oracle.moe_layer(x, b["wr"], k, **args)
            assert_close(y_out, gy, "moe block", terms=combine_terms(x, gids, gw, blk["_dl"]))
    rr, _, rids = oracle.decode_stack(synth.bits(x0), ob, EPS)
    for a, b in zip(ids, rids):
        for t in range(a.shape[0]):
            assert set(a[t]) == set(b[t])
    a, ref = bf16_to_f64(r), bf16_to_f64(rr)
    assert np.linalg.norm(a - ref) / np.linalg.norm(ref) <= 1e-2


def test_short_stack_pdl_is_bitwise_identical(stack):
    f = flint()
    blocks, x0, _ = stack
    r0, ids0 = run_stack(f, blocks, x0, 6, flags=0)
    r1, ids1 = run_stack(f, blocks, x0, 6, flags=f.FLINT_PDL)
    assert np.array_equal(r0, r1)
    for a, b in zip(ids0, ids1):
        assert np.array_equal(a, b)
