"""Phase trace of the fused MoE-layer kernel (flint_moe_layer) on the GPU.

Builds the phase-trace variant of the library (FLINT_PHASE_TRACE: thread 0 of
every CTA stamps %clock64 at the kernel's phase boundaries), runs a CUDA graph
of PDL-chained layer calls over `--layers` resident seeded layers (the
benchmark's setting: every call reads its experts from HBM), and prints, per
phase, the median and maximum over the CTAs of the calls traced, for the
shared-expert CTAs and the routed-expert CTAs separately, in thousands of SM
cycles.

    python -m nvfp4_moe_decode_sigmoid_gb300.phase_trace --tokens 1

Phases (stamp i to stamp i + 1):
  0 entry -> PDL wait passed      the static copies issued; waiting for the previous call
  1 -> x staged                   x read and converted (or the norm of the residual)
  2 -> router scores published    this CTA's router rows (bulk copy) times x
  3 -> routing known              all scores read, top-k, the work split, the first copies issued
  4 -> first chunk in             the first ring chunk's bytes landed
  5 -> gate/up done               the CTA's gate/up pairs, h published
  6 -> h staged                   the h of its down experts read (waits for the other CTAs)
  7 -> down done                  its down rows, d written
  8 -> arrivals                   the counts on its row blocks
  9 -> end                        the combine of the blocks it completed
"""
from __future__ import annotations

import argparse
import ctypes as C
import os
import statistics
import sys

import numpy as np

PHASES = ["wait for the previous call", "x staged", "router scores published", "routing, split, first copies",
          "first chunk in", "gate/up", "h of the down experts staged", "down", "arrivals", "combine"]
N_STAMPS, N_CALLS, N_CTAS = 16, 64, 256


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--tokens", type=int, default=1)
    p.add_argument("--routing", choices=["uniform", "zipf"], default="uniform")
    p.add_argument("--layers", type=int, default=32)
    p.add_argument("--calls", type=int, default=64, help="calls per graph (the trace keeps the last 64)")
    p.add_argument("--hidden", type=int, default=2048)
    p.add_argument("--experts", type=int, default=256)
    p.add_argument("--inter", type=int, default=512)
    p.add_argument("--top-k", type=int, default=6)
    args = p.parse_args(argv)

    from . import _build
    os.environ["FLINT_LIBRARY"] = _build.build(trace=True)
    import torch

    from . import flint as F
    from . import synth
    if "libflint_trace" not in F.LIBRARY_PATH:
        sys.exit("the binding was imported before the trace build was selected")
    read = F.raw_library().flint_phase_trace_read
    read.restype = C.c_longlong
    read.argtypes = [C.c_void_p, C.c_size_t]

    H, E, I, k, T = args.hidden, args.experts, args.inter, args.top_k, args.tokens
    layers = []
    for li in range(args.layers):
        L = synth.Layer(1000 + li, H=H, E=E, I=I, I_shared=I, device="cuda")
        s = L.shared
        layers.append(dict(router_w=L.router_w, routed=F.Experts.from_gguf(L.gate, L.up, L.down, L.ts, E, H, I),
                           shared=F.Experts.from_gguf(s["gate"], s["up"], s["down"], s["ts"].reshape(1, 3), 1, H, I),
                           x=synth.activations((1000 + li) * 31 + T, T, H, "cuda"),
                           ids=torch.empty((T, k), dtype=torch.int32, device="cuda"),
                           w=torch.empty((T, k), dtype=torch.float32, device="cuda"),
                           y=torch.empty((T, H), dtype=torch.bfloat16, device="cuda")))
        del L, s
    bias = synth.zipf_bias(7, E).cuda() if args.routing == "zipf" else None
    ws = torch.empty(F.flint_workspace_bytes(E, k, H, I, I), dtype=torch.uint8, device="cuda")
    F.flint_workspace_init(ws)

    def step(i):
        lay = layers[i % len(layers)]
        F.flint_moe_layer(lay["x"], lay["router_w"], k, lay["routed"], lay["shared"], lay["ids"], lay["w"], lay["y"],
                          ws, bias=bias, flags=F.FLINT_PDL)

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(len(layers)):
            step(i)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(args.calls):
                step(i)
        for _ in range(4):
            g.replay()
    torch.cuda.synchronize()
    assert F.flint_workspace_check(ws) == F.FLINT_OK, F.flint_last_error()

    buf = np.zeros(N_CALLS * N_CTAS * N_STAMPS, np.uint64)
    n = read(buf.ctypes.data_as(C.c_void_p), buf.size)
    assert n == buf.size, "reading the trace failed"
    tr = buf.reshape(N_CALLS, N_CTAS, N_STAMPS).astype(np.int64)
    G = torch.cuda.get_device_properties(0).multi_processor_count
    tr = tr[:, :G]
    calls = [c for c in range(N_CALLS) if np.all(tr[c, :, 15] == tr[c, 0, 15]) and tr[c, 0, 15] > 0]
    shared_role = (tr[:, :, 12] & 0xFF) == 1
    durations = {}  # (role, phase) -> list of cycles
    for c in calls:
        for cta in range(G):
            role = "shared" if shared_role[c, cta] else "routed"
            st = tr[c, cta, :11]
            for ph in range(10):
                durations.setdefault((role, ph), []).append(int(st[ph + 1] - st[ph]))
    # kernel span from the coarse global timer: first entry to last end of each call
    spans = [(tr[c, :, 14].max() - tr[c, :, 13].min()) / 1e3 for c in calls]
    print(f"## Fused layer phases: T = {T}, {args.routing} routing, {len(calls)} calls traced "
          f"({args.layers} resident layers, PDL-chained in one CUDA graph)\n")
    print("kcycles of the SM clock, median / max over the CTAs of all traced calls\n")
    print("| phase | shared-expert CTAs | routed-expert CTAs |")
    print("|---|---|---|")
    for ph in range(10):
        cells = []
        for role in ("shared", "routed"):
            v = durations.get((role, ph), [])
            cells.append(f"{statistics.median(v) / 1e3:.2f} / {max(v) / 1e3:.2f}" if v else "-")
        print(f"| {ph} {PHASES[ph]} | {cells[0]} | {cells[1]} |")
    tot = {role: [int(tr[c, cta, 10] - tr[c, cta, 1]) for c in calls for cta in range(G)
                  if (role == "shared") == bool(shared_role[c, cta])] for role in ("shared", "routed")}
    print(f"| after the wait, to the end | {statistics.median(tot['shared']) / 1e3:.2f} / "
          f"{max(tot['shared']) / 1e3:.2f} | {statistics.median(tot['routed']) / 1e3:.2f} / "
          f"{max(tot['routed']) / 1e3:.2f} |")
    print(f"\nCTAs: {int(shared_role[calls[0]].sum())} shared, {G - int(shared_role[calls[0]].sum())} routed; "
          f"call span on the global timer (first entry to last end, includes the wait for the previous call): "
          f"median {statistics.median(spans):.2f} us")


if __name__ == "__main__":
    main()
