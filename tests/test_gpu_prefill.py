"""GPU prefill (the MoE layer over many tokens on the tensor cores) against the
oracle: on every token whose top-k margin is at least 1e-3 the selected
experts must match, and on a sample of those tokens (seeded; at 8192 tokens
one covering every M-tile of the grouped GEMMs) the outputs must be within
the layer tolerance. Repeated runs must agree bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from flint_testlib import DeviceLayer, MARGIN, assert_close, bf16_to_f64, flint, terms_where_needed, combine_terms
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu


def run_prefill(dl, x, k, bias=None):
    f = flint()
    T, H = x.shape
    L = dl.L
    Is = L.Is if L.shared is not None else 0
    ws = torch.empty(f.flint_prefill_workspace_bytes(T, L.E, k, H, L.I, Is), dtype=torch.uint8, device="cuda")
    f.flint_workspace_init(ws)
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    f.flint_moe_prefill(x.cuda(), dl.router_w, k, dl.routed, dl.shared, ids, w, y, ws,
                        bias=None if bias is None else bias.cuda())
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    return ids.cpu().numpy(), w.cpu().numpy(), synth.bits(y)


def check_prefill(dl, x, k, n_sample, bias=None, seed=0):
    ids, w, y = run_prefill(dl, x, k, bias)
    T = x.shape[0]
    xb = synth.bits(x)
    wr = synth.bits(dl.L.router_w)
    b = None if bias is None else bias.numpy()
    rids, rw, s = oracle.router(xb, wr, k, b)
    ss = np.sort(s, axis=1)[:, ::-1]
    margin_ok = (ss[:, k - 1] - ss[:, k] >= MARGIN) if k < s.shape[1] else np.ones(T, bool)
    assert margin_ok.mean() > 0.5
    for t in np.nonzero(margin_ok)[0]:
        assert set(ids[t]) == set(rids[t]), f"token {t}"
        order = np.argsort(ids[t])
        np.testing.assert_allclose(w[t][order], rw[t][np.argsort(rids[t])], rtol=2e-5, atol=1e-7)
    assert np.all((ids >= 0) & (ids < dl.L.E))
    rng = np.random.default_rng(seed)
    cand = np.nonzero(margin_ok)[0]
    pick = np.sort(rng.choice(cand, size=min(n_sample, cand.size), replace=False))
    ref = oracle.moe_experts(xb[pick], rids[pick], rw[pick].astype(np.float32), **dl.oracle_args())
    terms = combine_terms(xb[pick], rids[pick], rw[pick], dl)
    assert_close(y[pick], ref, "prefill", terms=terms)
    return ids, w, y


@pytest.fixture(scope="module")
def small_layer():
    return DeviceLayer(synth.Layer(41, H=1024, E=16, I=256, I_shared=256))


@pytest.mark.parametrize("T,k", [(1, 6), (129, 6), (300, 4), (1000, 6)])
def test_small_prefill(small_layer, T, k):
    x = synth.activations(500 + T, T, 1024)
    check_prefill(small_layer, x, k, n_sample=12, seed=T)


def test_small_prefill_skewed_routing(small_layer):
    """A Zipf bias leaves some experts with no tokens (empty groups)."""
    bias = synth.zipf_bias(9, 16, s=2.0) * 3.0
    x = synth.activations(77, 400, 1024)
    ids, _, _ = check_prefill(small_layer, x, 2, n_sample=16, bias=bias, seed=3)
    assert len(set(ids.reshape(-1).tolist())) < 16


def test_small_prefill_is_deterministic(small_layer):
    x = synth.activations(78, 700, 1024)
    a = run_prefill(small_layer, x, 6)
    b = run_prefill(small_layer, x, 6)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_prefill_without_shared_expert():
    dl = DeviceLayer(synth.Layer(42, H=1024, E=32, I=256, I_shared=0, shared=False))
    x = synth.activations(79, 260, 1024)
    check_prefill(dl, x, 6, n_sample=12, seed=5)


@pytest.fixture(scope="module")
def full_layer():
    return DeviceLayer(synth.Layer(1007))


def test_full_prefill_8k_tokens(full_layer):
    """The prefill workload: 8192 tokens through one full-size layer. Ids and
    weights are checked on every token whose top-k margin is at least 1e-3.
    Outputs are checked on a sample that covers every 128-row M-tile of the
    grouped GEMMs: the kernel sorts each expert's (token, rank) pairs in token
    order, so one token from each 128-token run of an expert's token list (its
    last, so that the ragged tail tiles are in) covers the routed tiles, one
    token per 128 tokens covers the shared expert's and the router's, plus the
    first and last token. The oracle runs on all host cores (same bits)."""
    T, k = 8192, 6
    E = full_layer.L.E
    x = synth.activations(4096, T, 2048)
    ids, w, y = run_prefill(full_layer, x, k)
    assert np.all(np.isfinite(bf16_to_f64(y)))
    assert np.all((ids >= 0) & (ids < E))
    oracle.use_openmp(0)
    try:
        xb = synth.bits(x)
        rids, rw, s = oracle.router(xb, synth.bits(full_layer.L.router_w), k)
        ss = np.sort(s, axis=1)[:, ::-1]
        ok = ss[:, k - 1] - ss[:, k] >= MARGIN
        assert ok.mean() > 0.5
        for t in np.nonzero(ok)[0]:
            assert set(ids[t]) == set(rids[t]), f"token {t}"
            np.testing.assert_allclose(w[t][np.argsort(ids[t])], rw[t][np.argsort(rids[t])], rtol=2e-5,
                                       atol=1e-7)

        def last_ok(run):  # the last token of a run whose selection is certain
            good = run[ok[run]]
            return [int(good[-1])] if good.size else []

        pick = set(last_ok(np.array([0])) + last_ok(np.array([T - 1])))
        for e in range(E):
            toks = np.nonzero((rids == e).any(axis=1))[0]
            for j in range(0, toks.size, 128):
                pick.update(last_ok(toks[j:j + 128]))
        for j in range(0, T, 128):
            pick.update(last_ok(np.arange(j, min(T, j + 128))))
        pick = np.array(sorted(pick))
        assert pick.size > E  # (a token covers one tile of each of its k experts and of the shared expert)
        ref = oracle.moe_experts(xb[pick], rids[pick], rw[pick].astype(np.float32), **full_layer.oracle_args())
        terms = terms_where_needed(y[pick], ref, lambda r: combine_terms(xb[pick[r]], rids[pick[r]], rw[pick[r]],
                                                                        full_layer))
        assert_close(y[pick], ref, f"prefill 8k ({pick.size} tokens)", terms=terms)
    finally:
        oracle.use_openmp(-1)
