"""GPU router (GEMV + sigmoid top-k + renormalisation) against the oracle:
the selected experts bit-exact (inputs keep a top-k margin >= 1e-3), the
weights within FP32 rounding."""
import numpy as np
import pytest
import torch

import oracle
from flint_testlib import flint, margin_x
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu


def _run(x, wr, k, bias=None, flags=0):
    f = flint()
    T = x.shape[0]
    E = wr.shape[0]
    ws = torch.empty(f.flint_workspace_bytes(E, k, 0, 0, 0), dtype=torch.uint8, device="cuda")
    f.flint_workspace_init(ws)
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    b = bias.cuda() if bias is not None else None
    f.flint_moe_route(x.cuda(), wr.cuda(), k, ids, w, ws, bias=b, flags=flags)
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    return ids.cpu().numpy(), w.cpu().numpy()


def _compare(x, wr, k, bias=None, flags=0):
    ids, w = _run(x, wr, k, bias, flags)
    rids, rw, _ = oracle.router(synth.bits(x), synth.bits(wr), k, None if bias is None else bias.numpy())
    for t in range(x.shape[0]):
        assert set(ids[t]) == set(rids[t]), f"token {t}: {sorted(ids[t])} vs {sorted(rids[t])}"
        got = dict(zip(ids[t], w[t]))
        for e, we in zip(rids[t], rw[t]):
            assert abs(got[e] - we) <= 2e-6 * we + 1e-7
        assert abs(w[t].sum() - 1.0) < 1e-5
    return ids, w


@pytest.mark.parametrize("T", [1, 3, 8])
@pytest.mark.parametrize("E,k,H", [(256, 6, 2048), (16, 2, 256), (100, 8, 512), (8, 1, 1024), (1024, 6, 256)])
def test_route_matches_oracle(T, E, k, H):
    wr = synth.bf16_normal(E * 7 + H, (E, H), 0.02)
    x = margin_x(synth.bits(wr), T, H, k, None, seed=T * 31 + E)
    _compare(x, wr, k)


@pytest.mark.parametrize("T", [1, 8])
def test_route_with_zipf_bias(T):
    E, k, H = 256, 6, 2048
    wr = synth.bf16_normal(77, (E, H), 0.02)
    bias = synth.zipf_bias(5, E)
    x = margin_x(synth.bits(wr), T, H, k, bias.numpy(), seed=99)
    ids, _ = _compare(x, wr, k, bias)


def test_route_pdl_flag_gives_identical_results():
    f = flint()
    E, k, H, T = 256, 6, 2048, 8
    wr = synth.bf16_normal(3, (E, H), 0.02)
    x = margin_x(synth.bits(wr), T, H, k, None, seed=5)
    a = _run(x, wr, k, flags=0)
    b = _run(x, wr, k, flags=f.FLINT_PDL)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_route_all_equal_scores_pick_lowest_indices():
    E, k, H, T = 256, 6, 2048, 2
    wr = torch.zeros((E, H), dtype=torch.bfloat16)
    x = synth.activations(1, T, H)
    ids, w = _run(x, wr, k)
    assert np.array_equal(ids, np.tile(np.arange(k, dtype=np.int32), (T, 1)))
    assert np.allclose(w, 1.0 / k, atol=1e-7)


def test_route_repeated_calls_reuse_the_workspace():
    # the arrival counter must be back at zero after every call
    f = flint()
    E, k, H, T = 64, 4, 512, 4
    wr = synth.bf16_normal(8, (E, H), 0.02)
    x = margin_x(synth.bits(wr), T, H, k, None, seed=8)
    ws = torch.empty(f.flint_workspace_bytes(E, k, 0, 0, 0), dtype=torch.uint8, device="cuda")
    f.flint_workspace_init(ws)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    xc, wc = x.cuda(), wr.cuda()
    outs = []
    for _ in range(5):
        f.flint_moe_route(xc, wc, k, ids, w, ws, flags=f.FLINT_PDL)
        outs.append(ids.cpu().numpy().copy())
    assert all(np.array_equal(o, outs[0]) for o in outs)
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    assert int(ws[:4].view(torch.int32).item()) == 0
