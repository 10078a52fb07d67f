"""Helpers for the GPU parity tests: seeded layers on the device, inputs with
a guaranteed top-k margin, and the tolerance check."""
import numpy as np
import torch

import oracle
from nvfp4_moe_decode_sigmoid_gb300 import synth

# Layer outputs: relative L2 error <= 1e-2 and per element
# |gpu - ref| <= 3e-2 * (|ref| + 1e-2) against the oracle.
REL_L2 = 1e-2
ELEM_A, ELEM_B = 3e-2, 1e-2
MARGIN = 1e-3


def flint():
    from nvfp4_moe_decode_sigmoid_gb300 import _build
    _build.build()
    from nvfp4_moe_decode_sigmoid_gb300 import flint as f
    return f


def bf16_to_f64(bits):
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_ulp(v):
    """One unit in the last place of bf16 at magnitude |v| (8 significant bits)."""
    mag = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(mag)) - 7)


def assert_close(y_gpu_bits, y_ref_bits, what="", terms=None):
    """The layer tolerance: relative L2 error <= REL_L2 and per element
    |gpu - ref| <= ELEM_A (|ref| + ELEM_B).

    terms (optional, [T, H], from combine_terms): per output element the
    magnitude sum_j |w_j d_j| + |d_shared| of the terms the combine adds. The
    GPU and the oracle both compute in FP32 with bf16 at the stated rounding
    points, in different summation orders; near a bf16 rounding boundary
    their g, u, h or d then round one ulp apart, and a few such steps can move
    y by a few bf16 ulps of the terms. Where the terms cancel (|y| much
    smaller than them) that exceeds the bound relative to |y| without an
    error on either side: an evaluation of the oracle's own definition in
    another FP32 order (tests/test_oracle_tolerance.py) does so. With
    `terms`, an element outside the per-element bound still passes if its
    error is within the same bound relative to the terms, ELEM_A (terms +
    ELEM_B), and such elements must be rare (at most 0.1 %, at least one
    allowed); relative L2 still holds for all."""
    a, r = bf16_to_f64(y_gpu_bits), bf16_to_f64(y_ref_bits)
    assert np.all(np.isfinite(a)), f"{what}: non-finite GPU output"
    rel = np.linalg.norm(a - r) / max(np.linalg.norm(r), 1e-30)
    assert rel <= REL_L2, f"{what}: relative L2 error {rel:.3e} > {REL_L2}"
    err = np.abs(a - r)
    bad = err > ELEM_A * (np.abs(r) + ELEM_B)
    if terms is not None and bad.any():
        cancel = bad & (err <= ELEM_A * (np.asarray(terms, np.float64) + ELEM_B))
        assert cancel.sum() <= max(1, 1e-3 * bad.size), f"{what}: {int(cancel.sum())} cancellation outliers"
        bad = bad & ~cancel
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside tolerance, e.g. gpu {a[bad][:4]} ref {r[bad][:4]}"
    return rel


def terms_where_needed(y_gpu_bits, y_ref_bits, terms_of_rows):
    """The `terms` argument of assert_close, computed (by terms_of_rows(rows))
    only for the rows (tokens) that have an element outside the per-element
    bound; 0 elsewhere, where no element needs it."""
    a, r = bf16_to_f64(y_gpu_bits), bf16_to_f64(y_ref_bits)
    rows = np.nonzero((np.abs(a - r) > ELEM_A * (np.abs(r) + ELEM_B)).any(axis=1))[0]
    terms = np.zeros(r.shape)
    if rows.size:
        terms[rows] = terms_of_rows(rows)
    return terms


def combine_terms(x_bits, ids, weights, dl):
    """Per token and output row: sum_j |w_j d_j| + |d_shared|, the magnitude of
    the terms the combine adds, from the oracle's per-expert outputs."""
    args = dl.oracle_args()
    L = dl.L
    H, I = L.H, L.I
    x_bits = np.asarray(x_bits, np.uint16)
    T, k = ids.shape
    per = lambda a, e: np.ascontiguousarray(a.reshape(L.E, -1)[e])  # noqa: E731
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            ts = args["ts"][e] if args["ts"] is not None else (1.0, 1.0, 1.0)
            _, _, _, d = oracle.expert(x_bits[t], per(args["gate"], e), per(args["up"], e),
                                       per(args["down"], e), H, I, ts=ts, wdtype=args["wdtype"])
            out[t] += np.abs(float(weights[t, j]) * bf16_to_f64(d))
        sh = args["shared"]
        if sh is not None:
            ts = sh["ts"] if sh["ts"] is not None else (1.0, 1.0, 1.0)
            _, _, _, d = oracle.expert(x_bits[t], sh["gate"].reshape(-1), sh["up"].reshape(-1),
                                       sh["down"].reshape(-1), H, sh["I"], ts=ts, wdtype=args["wdtype"])
            out[t] += np.abs(bf16_to_f64(d))
    return out




def margin_x(router_bits, T, H, k, bias, seed, margin=MARGIN):
    """Seeded tokens, each resampled until its k-th and (k+1)-th sigmoid scores
    (oracle, FP32 decision precision) differ by at least `margin`."""
    rows = []
    E = router_bits.shape[0]
    for t in range(T):
        rep = 0
        while True:
            x = synth.activations(seed * 100003 + t * 1009 + rep, 1, H)
            if k >= E:
                break
            _, _, s = oracle.router(synth.bits(x), router_bits, k, bias)
            ss = np.sort(s[0])[::-1]
            if ss[k - 1] - ss[k] >= margin:
                break
            rep += 1
        rows.append(x)
    return torch.cat(rows)


class DeviceLayer:
    """A synth.Layer (drawn on the CPU) copied to the GPU and repacked there."""

    def __init__(self, L: synth.Layer):
        f = flint()
        self.L = L
        dev = "cuda"
        self.router_w = L.router_w.to(dev)
        self.shared = None
        if L.wdtype == "nvfp4":
            self.routed = f.Experts.from_gguf(L.gate.to(dev), L.up.to(dev), L.down.to(dev), L.ts, L.E, L.H, L.I)
            if L.shared is not None:
                s = L.shared
                self.shared = f.Experts.from_gguf(s["gate"].to(dev), s["up"].to(dev), s["down"].to(dev),
                                                  s["ts"].reshape(1, 3), 1, L.H, s["I"])
        else:
            self.routed = f.Experts.from_bf16(L.gate.to(dev), L.up.to(dev), L.down.to(dev), L.E, L.H, L.I,
                                              None if L.ts is None else L.ts.to(dev))
            if L.shared is not None:
                s = L.shared
                self.shared = f.Experts.from_bf16(s["gate"].to(dev), s["up"].to(dev), s["down"].to(dev), 1, L.H,
                                                  s["I"], None if s["ts"] is None else s["ts"].reshape(1, 3).to(dev))
        torch.cuda.synchronize()

    def oracle_args(self):
        L = self.L
        if L.wdtype == "nvfp4":
            w = lambda t: t.numpy()  # noqa: E731
            wdtype = oracle.W_NVFP4
        else:
            w = synth.bits
            wdtype = oracle.W_BF16
        opt = lambda t: None if t is None else t.numpy()  # noqa: E731
        sh = None
        if L.shared is not None:
            s = L.shared
            sh = dict(gate=w(s["gate"]), up=w(s["up"]), down=w(s["down"]), ts=opt(s["ts"]), I=s["I"])
        return dict(E=L.E, I=L.I, gate=w(L.gate), up=w(L.up), down=w(L.down), ts=opt(L.ts), shared=sh,
                    wdtype=wdtype)

    def workspace(self, k):
        f = flint()
        Is = self.L.Is if self.L.shared is not None else 0
        ws = torch.empty(f.flint_workspace_bytes(self.L.E, k, self.L.H, self.L.I, Is), dtype=torch.uint8, device="cuda")
        f.flint_workspace_init(ws)
        return ws
