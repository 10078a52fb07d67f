"""Phase trace of the fused MoE-layer kernel (flint_moe_layer) on the GPU.

Builds the phase-trace variant of the library (FLINT_PHASE_TRACE: thread 0 of
every CTA stamps %clock64 at the kernel's phase boundaries), runs a CUDA graph
of PDL-chained layer calls over `--layers` resident seeded layers (the
benchmark's setting: every call reads its experts from HBM), and prints, per
phase, the median and maximum over the CTAs of the calls traced, for the
shared-expert CTAs and the routed-expert CTAs separately, in thousands of SM
cycles.

    python -m nvfp4_moe_decode_sigmoid_gb300.phase_trace --tokens 1
    python -m nvfp4_moe_decode_sigmoid_gb300.phase_trace --tokens 8 --path decode

--path decode traces flint_moe_decode as one kernel (the routing given: each
call follows flint_moe_route on the same x, PDL-chained) instead of
flint_moe_layer; its routed CTAs have no router rows or score exchange, and
"ids read" replaces those intervals.

Intervals (between the kernel's stamps; "-" where a group of CTAs has none):
  wait for the previous call      entry to the PDL wait's return (static copies issued)
  x staged                        x read and converted (or the norm of the residual)
  router scores published         this CTA's router rows (bulk copy) times x, the count raised
  all scores in                   waiting until every router row is published
  top-k                           one warp per token, its scores read from L2
  routing view                    the distinct experts and their tokens
  split                           this CTA's ranges (cost split) and runs
  first copies                    the plan shared, each warp's first ring copies issued
  first chunk in                  the first ring item's bytes landed
  gate/up                         the CTA's gate/up pairs, h written and counted
  h of the down experts staged    waits for the other CTAs' h of those experts
  down                            its down rows, d written
  at the end: ...                 the shared group's routing steps, for the combine weights
  arrivals                        the counts on its row blocks
  combine                         the blocks it completed
One token (down split by output rows):
  routing (shared group)          the shared group's routing, after its gate/up
  h of the down experts staged    here: every pair published, all of h staged
  down                            the CTA's rows of every expert's down GEMV
  after the down items            its rows of y (with more tokens: arrivals and combine)
"""
from __future__ import annotations

import argparse
import ctypes as C
import os
import statistics
import sys

import numpy as np

# (name, from stamp, to stamp); the stamps the kernel takes (see layer.cu)
INTERVALS = [("wait for the previous call", 0, 1, "all"), ("x staged", 1, 2, "all"),
             ("ids read (decode)", 3, 13, "decode"),
             ("router scores published", 2, 3, "routed"), ("all scores in", 3, 11, "routed"),
             ("top-k", 12, 13, "routed"), ("routing view", 13, 14, "routed"), ("split", 14, 19, "routed"),
             ("first copies", 19, 4, "routed"), ("first chunk in", 4, 5, "all"), ("gate/up", 5, 6, "all"),
             ("h of the down experts staged", 6, 7, "all"), ("down", 7, 8, "all"),
             ("at the end: all scores in", 8, 15, "shared"), ("at the end: top-k", 16, 17, "shared"),
             ("at the end: routing view", 17, 18, "shared"), ("arrivals", 18, 9, "shared"),
             ("arrivals", 8, 9, "routed"), ("combine", 9, 10, "all"),
             ("one token: routing (shared group, after its gate/up)", 6, 43, "shared"),
             ("after the down items, to the end", 8, 10, "all"),
             ("after the wait, to the end", 1, 10, "all")]
# The one-token kernel (layer_one_kernel, marked 2 in the low byte of stamp
# 28): every CTA holds a share of every step, so one column.
INTERVALS_ONE = [("wait for the previous call", 0, 1), ("x staged", 1, 2),
                 ("router row published (fence, count)", 2, 3), ("x staged to all scores in", 2, 5),
                 ("top-k warp: waiting for the scores", 4, 5), ("top-k", 5, 6),
                 ("routing shared with the CTA", 6, 7), ("routed copies issued", 7, 8),
                 ("first routed pair done", 8, 9), ("routing to every pair done, h written", 7, 10),
                 ("all pairs published (h exchange)", 10, 11), ("all of h staged", 11, 12),
                 ("down rows of every expert", 12, 13), ("rows of y", 13, 14),
                 ("after the wait, to the end", 1, 14)]
N_STAMPS, N_CALLS, N_CTAS = 48, 64, 256


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
    p.add_argument("--path", choices=["layer", "decode", "block"], default="layer")
    p.add_argument("--dump", default=None, help="also save the raw stamps ([calls][CTAs][stamps]) to this .npy file")
    args = p.parse_args(argv)

    from . import _build
    if "trace" not in os.path.basename(os.environ.get("FLINT_LIBRARY", "")):  # a trace build chosen by the caller
        os.environ["FLINT_LIBRARY"] = _build.build(trace=True)
    import torch

    from . import flint as F
    from . import synth
    if "trace" not in os.path.basename(F.LIBRARY_PATH):
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

    # block: pre-norm blocks chained as in a decode stack (each block's y is the
    # next one's y_prev; the residual stream ping-pongs between two buffers)
    res = [synth.activations(5, T, H, "cuda"), torch.empty((T, H), dtype=torch.bfloat16, device="cuda")]
    ys = [torch.zeros((T, H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]

    def step(i):
        lay = layers[i % len(layers)]
        if args.path == "block":
            F.flint_moe_block(res[i % 2], lay["router_w"], k, lay["routed"], lay["shared"], lay["ids"], lay["w"],
                              ys[i % 2], ws, y_prev=ys[(i + 1) % 2] if i else None, residual_out=res[(i + 1) % 2],
                              bias=bias, flags=F.FLINT_PDL)
            return
        if args.path == "decode":
            F.flint_moe_route(lay["x"], lay["router_w"], k, lay["ids"], lay["w"], ws, bias=bias, flags=F.FLINT_PDL)
            F.flint_moe_decode(lay["x"], lay["ids"], lay["w"], lay["routed"], lay["shared"], lay["y"], ws,
                               flags=F.FLINT_PDL | F.FLINT_PDL_AFTER_ROUTE)
            return
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
    if args.dump:
        np.save(args.dump, tr)
    calls = [c for c in range(N_CALLS) if np.all(tr[c, :, 31] == tr[c, 0, 31]) and tr[c, 0, 31] > 0]
    if calls and np.all((tr[calls, :, 28] & 0xFF) == 2):
        return report_one(args, tr, calls, G)
    shared_role = (tr[:, :, 28] & 0xFF) == 1
    cells = {}  # (role, interval) -> list of cycles
    for c in calls:
        for cta in range(G):
            role = "shared" if shared_role[c, cta] else "routed"
            st = tr[c, cta]
            for n, (_, a, b, who) in enumerate(INTERVALS):
                if who == "decode":
                    who = "routed" if args.path == "decode" else None
                elif args.path == "decode" and a in (2, 35) and b in (3, 36, 37):
                    who = None  # no router rows on this path
                if who in ("all", role) and st[a] and st[b]:
                    cells.setdefault((role, n), []).append(int(st[b] - st[a]))
    spans = [(tr[c, :, 30].max() - tr[c, :, 29].min()) / 1e3 for c in calls]
    # spread over the CTAs of one call (global timer, coarse): entries, score publications
    entry_spread = [(tr[c, :, 29].max() - tr[c, :, 29].min()) / 1e3 for c in calls]
    pub = [tr[c, tr[c, :, 26] > 0, 26] for c in calls]
    pub_spread = [(p.max() - p.min()) / 1e3 for p in pub if p.size]
    what = {"layer": "Fused layer", "block": "Fused pre-norm blocks chained",
            "decode": "One-kernel decode (routing given, after the router)"}[args.path]
    print(f"## {what} phases: T = {T}, {args.routing} routing, {len(calls)} calls traced "
          f"({args.layers} resident layers, PDL-chained in one CUDA graph)\n")
    print("kcycles of the SM clock, median / max over the CTAs of all traced calls\n")
    print("| interval | shared-expert CTAs | routed-expert CTAs |")
    print("|---|---|---|")
    for n, (name, _, _, _) in enumerate(INTERVALS):
        row = []
        for role in ("shared", "routed"):
            v = cells.get((role, n), [])
            row.append(f"{statistics.median(v) / 1e3:.2f} / {max(v) / 1e3:.2f}" if v else "-")
        if row != ["-", "-"]:
            print(f"| {name} | {row[0]} | {row[1]} |")
    # warp 0 of each CTA: its gate/up items' waits for bytes, arithmetic, epilogue and refill; the
    # spread of the warps' ends of the gate/up loop
    med = lambda v: statistics.median(v) / 1e3
    for role in ("shared", "routed"):
        sel = [tr[c, cta] for c in calls for cta in range(G) if (role == "shared") == bool(shared_role[c, cta])]
        if not sel:
            continue
        print(f"\n{role}, warp 0 over its {statistics.median([int(st[23]) & 0xFFFF for st in sel]):.0f} gate/up "
              f"items (median kcycles): waits {med([int(st[20]) for st in sel]):.2f}, arithmetic "
              f"{med([int(st[21]) for st in sel]):.2f}, epilogue and refill {med([int(st[22]) for st in sel]):.2f}; "
              f"over its {statistics.median([(int(st[23]) >> 16) & 0xFFFF for st in sel]):.0f} down items waits "
              f"{med([int(st[23]) >> 32 for st in sel]):.2f}; warps' gate/up ends: last - first "
              f"{med([int(st[25] - st[24]) for st in sel]):.2f}, last - stamp 5 "
              f"{med([int(st[25] - st[5]) for st in sel if st[5]]):.2f}")
    n_sh = int(shared_role[calls[0]].sum())
    print(f"\nCTAs: {n_sh} shared, {G - n_sh} routed. On the global timer (coarse), median over the calls: "
          f"call span (first entry to last end, with the wait for the previous call) "
          f"{statistics.median(spans):.2f} us; spread of the CTAs' entries {statistics.median(entry_spread):.2f} us; "
          + (f"spread of their router-score publications {statistics.median(pub_spread):.2f} us" if pub_spread
             else "no router-score publications"))


def report_one(args, tr, calls, G):
    """The one-token kernel's intervals, median / max over all CTAs of the calls."""
    what = {"layer": "One-token layer kernel", "block": "One-token kernel, pre-norm blocks chained",
            "decode": "One-token kernel, routing given (after the router)"}[args.path]
    print(f"## {what} phases: {args.routing} routing, {len(calls)} calls traced "
          f"({args.layers} resident layers, PDL-chained in one CUDA graph)\n")
    print("kcycles of the SM clock, median / max over the CTAs of all traced calls\n")
    print("| interval | all CTAs |")
    print("|---|---|")
    for name, a, b in INTERVALS_ONE:
        if args.path == "decode":  # the routing given: no router rows, scores or top-k
            if (a, b) in ((2, 3), (4, 5), (5, 6)):
                continue
            name = {"x staged to all scores in": "ids and weights read"}.get(name, name)
        v = [int(tr[c, cta, b] - tr[c, cta, a]) for c in calls for cta in range(G) if tr[c, cta, a] and tr[c, cta, b]]
        if v:
            print(f"| {name} | {statistics.median(v) / 1e3:.2f} / {max(v) / 1e3:.2f} |")
    spans = [(tr[c, :, 30].max() - tr[c, :, 29].min()) / 1e3 for c in calls]
    entry = [(tr[c, :, 29].max() - tr[c, :, 29].min()) / 1e3 for c in calls]
    pub = [tr[c, tr[c, :, 26] > 0, 26] for c in calls]
    pub_spread = [(p.max() - p.min()) / 1e3 for p in pub if p.size]
    # consecutive calls n, n + 1: the first entry of n + 1 against the last end of n, and the last entry of
    # n + 1 against the last end of n (negative: overlap)
    by_no = {int(tr[c, 0, 31]): c for c in calls}
    first_gap, last_gap = [], []
    for n, c in by_no.items():
        if n + 1 in by_no:
            c1 = by_no[n + 1]
            first_gap.append((tr[c1, :, 29].min() - tr[c, :, 30].max()) / 1e3)
            last_gap.append((tr[c1, :, 29].max() - tr[c, :, 30].max()) / 1e3)
    print(f"\nOn the global timer (coarse), median over the calls: call span (first entry to last end, with the "
          f"wait for the previous call) {statistics.median(spans):.2f} us; spread of the CTAs' entries "
          f"{statistics.median(entry):.2f} us; spread of their first router-row publications "
          f"{statistics.median(pub_spread) if pub_spread else float('nan'):.2f} us")
    if first_gap:
        print(f"Between consecutive calls: first entry of the next call minus last end of this one "
              f"{statistics.median(first_gap):.2f} us, last entry of the next minus last end of this one "
              f"{statistics.median(last_gap):.2f} us ({len(first_gap)} pairs)")


if __name__ == "__main__":
    main()
