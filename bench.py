"""Benchmark: decode step of one Flint-style NVFP4 MoE layer on GB300.

A step is one pass of the whole hot path (router GEMV + sigmoid top-6 ->
gate/up GEMV + SiLU -> down GEMV + weighted combine with the shared expert)
over one batch of T tokens, through the C ABI: one flint_moe_layer launch per
layer (all steps in one cooperative kernel), PDL-chained to the previous
layer's, replayed from a CUDA graph. The three-kernel chain (flint_moe_route
-> flint_moe_decode) is timed on the same workload for comparison. Weights of `--layers` distinct seeded layers stay resident in HBM
and the steps cycle through them, so every step reads its experts from HBM
(the rotation's reuse distance is far larger than the 129 MB L2).

value = algorithmic bytes / time, in GB/s: router weights + the packed codes,
scales and tensor scales of the distinct selected experts + the shared expert
+ x + y, per step, as the routing of each layer actually selects them.

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle on the
same workload instead (a deliberately slow baseline).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

H, E, I, I_SHARED, TOPK = 2048, 256, 512, 512, 6
ROUTER_BYTES = E * H * 2
WORKLOADS = {
    # name: (tokens, routing)
    "moe-layer-b8-uniform": (8, "uniform"),
    "moe-layer-b1": (1, "uniform"),
    "moe-layer-b8-zipf": (8, "zipf"),
}
DEFAULT_WORKLOAD = "moe-layer-b8-uniform"
METRIC = "NVFP4 MoE-layer decode achieved HBM GB/s (algorithmic bytes / layer time)"
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (context beside the measured copy bandwidth)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=65536)
    p.add_argument("--warmup", type=int, default=256)
    p.add_argument("--impl", choices=["flint", "reference"], default="flint")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    p.add_argument("--layers", type=int, default=32)
    p.add_argument("--graph-steps", type=int, default=64)
    p.add_argument("--no-extra", action="store_true", help="skip the other two batch/routing workloads")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-bf16", action="store_true", help="skip the BF16-expert variant")
    p.add_argument("--no-stack", action="store_true", help="skip the 49-block decode stack")
    p.add_argument("--no-prefill", action="store_true", help="skip the 8192-token prefill")
    p.add_argument("--prefill-only", action="store_true",
                   help="only time the 8192-token prefill (one JSON line of its own; for profiling)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def replica_max(v: float, world: int, device: str) -> float:
    """The largest of the ranks' values (the slowest replica's time); every
    rank gets it. The ranks are independent replicas: this all-reduce of one
    number is the only exchange between them."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(bytes_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job GB/s: the bytes every replica processed over the slowest time."""
    return bytes_per_rank * world / (ms_max * 1e-3) / 1e9


def expert_bytes():
    from nvfp4_moe_decode_sigmoid_gb300 import flint as F
    gu = 2 * I * F.flint_nvfp4_row_stride(H)
    dn = H * F.flint_nvfp4_row_stride(I)
    return gu, dn


def step_bytes(n_distinct: int, T: int, with_bias: bool) -> int:
    gu, dn = expert_bytes()
    per_expert = gu + dn + 3 * 4  # codes + scales + the three FP32 tensor scales
    return ROUTER_BYTES + (E * 4 if with_bias else 0) + (n_distinct + 1) * per_expert + 2 * T * H * 2


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.dev), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "power_w_max": max(r["power"] for r in rows), "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class Model:
    """`n_layers` seeded MoE layers resident on the device: NVFP4 experts
    repacked to the kernel layout, or (wdtype "bf16") the 16-bit variant."""

    def __init__(self, n_layers: int, device, wdtype: str = "nvfp4"):
        import torch
        from nvfp4_moe_decode_sigmoid_gb300 import flint as F
        from nvfp4_moe_decode_sigmoid_gb300 import synth
        self.wdtype = wdtype
        self.layers = []
        for li in range(n_layers):
            L = synth.Layer(1000 + li, H=H, E=E, I=I, I_shared=I_SHARED, device=device, wdtype=wdtype)
            s = L.shared
            if wdtype == "nvfp4":
                routed = F.Experts.from_gguf(L.gate, L.up, L.down, L.ts, E, H, I)
                shared = F.Experts.from_gguf(s["gate"], s["up"], s["down"], s["ts"].reshape(1, 3), 1, H, I_SHARED)
            else:
                routed = F.Experts.from_bf16(L.gate, L.up, L.down, E, H, I)
                shared = F.Experts.from_bf16(s["gate"], s["up"], s["down"], 1, H, I_SHARED)
            self.layers.append(dict(router_w=L.router_w, routed=routed, shared=shared, seed=1000 + li))
            del L, s
            torch.cuda.synchronize()
        # each layer pulls the next one's router and shared expert into L2
        # before its PDL wait (static weights, as in a model's layer chain)
        for li, lay in enumerate(self.layers):
            nx = self.layers[(li + 1) % n_layers]
            lay["next_pf"] = F.l2_prefetch(nx["router_w"], nx["shared"].gate_up, nx["shared"].down)
        self.ws = torch.empty(F.flint_workspace_bytes(E, TOPK, H, I, I_SHARED), dtype=torch.uint8, device=device)
        F.flint_workspace_init(self.ws)
        # sized without the hidden size: flint_moe_decode runs as two kernels on it
        self.ws_small = torch.empty(F.flint_workspace_bytes(E, TOPK, 0, I, I_SHARED), dtype=torch.uint8,
                                    device=device)
        F.flint_workspace_init(self.ws_small)

    def step_bytes(self, n_distinct: int, T: int, with_bias: bool) -> int:
        if self.wdtype == "nvfp4":
            return step_bytes(n_distinct, T, with_bias)
        per_expert = 3 * I * H * 2  # bf16 gate, up, down; no tensor scales
        return ROUTER_BYTES + (E * 4 if with_bias else 0) + (n_distinct + 1) * per_expert + 2 * T * H * 2


def make_inputs(model, T, routing, device):
    import torch
    from nvfp4_moe_decode_sigmoid_gb300 import synth
    bias = synth.zipf_bias(7, E).to(device) if routing == "zipf" else None
    per = []
    for li, lay in enumerate(model.layers):
        per.append(dict(x=synth.activations(lay["seed"] * 31 + T, T, H, device),
                        ids=torch.empty((T, TOPK), dtype=torch.int32, device=device),
                        w=torch.empty((T, TOPK), dtype=torch.float32, device=device),
                        y=torch.empty((T, H), dtype=torch.bfloat16, device=device)))
    return bias, per


def run_step(F, model, inp, li, bias, flags, path="fused"):
    """One layer step: the fused kernel ("fused"), or the router then
    flint_moe_decode: one cooperative kernel on the full workspace ("chain"),
    gate/up and down kernels on one sized without the hidden size ("chain3")."""
    lay, io = model.layers[li], inp[li]
    if path == "fused":
        F.flint_moe_layer(io["x"], lay["router_w"], TOPK, lay["routed"], lay["shared"], io["ids"], io["w"], io["y"],
                          model.ws, bias=bias, flags=flags, next=lay["next_pf"])
        return
    ws = model.ws_small if path == "chain3" else model.ws
    F.flint_moe_route(io["x"], lay["router_w"], TOPK, io["ids"], io["w"], ws, bias=bias, flags=flags)
    dflags = flags | (F.FLINT_PDL_AFTER_ROUTE if flags & F.FLINT_PDL else 0)
    F.flint_moe_decode(io["x"], io["ids"], io["w"], lay["routed"], lay["shared"], io["y"], ws, flags=dflags)


def measure_workload(F, model, name, steps, warmup, graph_steps, sync_all, device_index, with_clocks=True,
                     path="fused"):
    import torch
    T, routing = WORKLOADS[name]
    nl = len(model.layers)
    bias, inp = make_inputs(model, T, routing, "cuda")
    flags = F.FLINT_PDL
    for s in range(max(warmup, nl)):
        run_step(F, model, inp, s % nl, bias, flags, path)
    torch.cuda.synchronize()
    assert F.flint_workspace_check(model.ws) == F.FLINT_OK
    assert F.flint_workspace_check(model.ws_small) == F.FLINT_OK
    # distinct experts each layer's routing selects -> algorithmic bytes per step
    distinct = [len(set(io["ids"].cpu().numpy().reshape(-1).tolist())) for io in inp]
    bytes_per_layer = [model.step_bytes(d, T, bias is not None) for d in distinct]

    stream = torch.cuda.Stream()
    R = max(1, min(graph_steps, steps))
    graphs = []
    with torch.cuda.stream(stream):
        for count, start in ((R, 0), (steps % R, 0)):
            if count == 0:
                continue
            g = torch.cuda.CUDAGraph()
            # offset so that consecutive replays continue the layer rotation
            with torch.cuda.graph(g, stream=stream):
                for s in range(count):
                    run_step(F, model, inp, (start + s) % nl, bias, flags, path)
            graphs.append((g, count))
    main_g, main_n = graphs[0]
    reps = steps // R
    tail = graphs[1] if len(graphs) > 1 else None
    # warm the graphs (replay() launches on the current stream: keep it `stream`)
    with torch.cuda.stream(stream):
        for _ in range(2):
            main_g.replay()
    torch.cuda.synchronize()

    total_bytes = 0
    for r in range(reps):
        total_bytes += sum(bytes_per_layer[s % nl] for s in range(R))
    if tail:
        total_bytes += sum(bytes_per_layer[s % nl] for s in range(tail[1]))

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device_index) if with_clocks else None
    if sampler:
        sampler.__enter__()
    sync_all()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            main_g.replay()
        if tail:
            tail[0].replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    sync_all()
    if sampler:
        sampler.__exit__(None, None, None)
    ms = ev0.elapsed_time(ev1)
    assert F.flint_workspace_check(model.ws) == F.FLINT_OK
    return dict(T=T, routing=routing, ms=ms, steps=steps, bytes=total_bytes,
                mean_distinct=sum(distinct) / len(distinct), clocks=sampler.summary() if sampler else None,
                bytes_per_step_mean=total_bytes / steps)


def measure_bf16(F, nvfp4_model, args, sync_all, dev_index, n_layers=6):
    """The BF16-weight variant of the same layer (router -> gate/up -> down,
    three PDL-chained kernels; the one-kernel layer and decode are NVFP4-only),
    at T = 1 and T = 8, beside the NVFP4 three-kernel chain on the same
    workloads.
    `n_layers` BF16 layers (1.5 GB each) rotate, so every step reads HBM."""
    import torch
    bmodel = Model(n_layers, "cuda", "bf16")
    peak, _ = load_peaks()
    out = {}
    for name in ("moe-layer-b1", "moe-layer-b8-uniform"):
        steps = max(512, min(4096, args.steps // 8))
        r = measure_workload(F, bmodel, name, steps, args.warmup, args.graph_steps, sync_all, dev_index,
                             with_clocks=False, path="chain")
        q = measure_workload(F, nvfp4_model, name, steps, args.warmup, args.graph_steps, sync_all, dev_index,
                             with_clocks=False, path="chain3")
        gbs = r["bytes"] / (r["ms"] * 1e-3) / 1e9
        out[name] = dict(us_per_layer=round(r["ms"] * 1e3 / r["steps"], 3), gb_s=round(gbs, 1),
                         frac_of_peak=round(gbs / peak, 4), bytes_per_step=r["bytes_per_step_mean"],
                         mean_distinct_experts=r["mean_distinct"],
                         nvfp4_chain_us_per_layer=round(q["ms"] * 1e3 / q["steps"], 3),
                         nvfp4_chain_bytes_per_step=q["bytes_per_step_mean"])
    del bmodel
    torch.cuda.empty_cache()
    out["path"] = "flint_moe_route -> flint_moe_decode (bf16 gate/up, bf16 down), PDL, CUDA graph"
    out["layers_rotated"] = n_layers
    return out


DENSE_F, N_DENSE, N_MOE = 6144, 2, 47


class Stack:
    """The decode stack of the model: N_DENSE dense SwiGLU MLP blocks
    (H -> DENSE_F -> H, NVFP4) then N_MOE MoE blocks, each seeded (block b from
    seed 1000 + b), resident on the device; residual add + RMSNorm (eps 1e-6,
    gamma 1) ahead of every block and once after the last."""

    def __init__(self, device):
        import torch
        from nvfp4_moe_decode_sigmoid_gb300 import flint as F
        from nvfp4_moe_decode_sigmoid_gb300 import synth
        self.dense, self.moe = [], []
        for b in range(N_DENSE):
            seed = 1000 + b
            gu = synth.gguf_nvfp4(synth._mix(seed, 20), 1, 2 * DENSE_F, H, device)
            dn = synth.gguf_nvfp4(synth._mix(seed, 21), 1, H, DENSE_F, device)
            ts = synth.tensor_scales(synth._mix(seed, 22), (3,), device)
            self.dense.append((F.Packed.from_gguf(gu, 2 * DENSE_F, H, ts[:2].contiguous()),
                               F.Packed.from_gguf(dn, H, DENSE_F, ts[2:].contiguous())))
            del gu, dn
        for b in range(N_DENSE, N_DENSE + N_MOE):
            L = synth.Layer(1000 + b, H=H, E=E, I=I, I_shared=I_SHARED, device=device)
            s = L.shared
            self.moe.append(dict(router_w=L.router_w,
                                 routed=F.Experts.from_gguf(L.gate, L.up, L.down, L.ts, E, H, I),
                                 shared=F.Experts.from_gguf(s["gate"], s["up"], s["down"], s["ts"].reshape(1, 3), 1,
                                                            H, I_SHARED)))
            del L, s
            torch.cuda.synchronize()
        for i, lay in enumerate(self.moe):  # each block pulls the next one's static weights into L2
            nx = self.moe[i + 1] if i + 1 < len(self.moe) else None
            lay["next_pf"] = F.l2_prefetch(nx["router_w"], nx["shared"].gate_up, nx["shared"].down) if nx else None
        self.ws = torch.empty(F.flint_workspace_bytes(E, TOPK, H, I, I_SHARED), dtype=torch.uint8, device=device)
        F.flint_workspace_init(self.ws)

    def dense_bytes(self):
        from nvfp4_moe_decode_sigmoid_gb300 import flint as F
        return (2 * DENSE_F * F.flint_nvfp4_row_stride(H) + H * F.flint_nvfp4_row_stride(DENSE_F) + 12)

    def step(self, F, io, flags):
        """One decode step of T tokens: 2 x (norm, SwiGLU GEMV, GEMV) + N_MOE
        fused blocks + the final residual add and norm."""
        r, y, x, h, ids, w = io["r"], io["y"], io["x"], io["h"], io["ids"], io["w"]
        src, nxt, y_prev = io["x0"], 0, None  # the embedding x0 is only read
        for b, (Wgu, Wdn) in enumerate(self.dense):
            if y_prev is None:
                F.flint_residual_rmsnorm(src, x, flags=flags)
            else:
                F.flint_residual_rmsnorm(src, x, y_prev=y_prev, residual_out=r[nxt], flags=flags)
                src, nxt = r[nxt], 1 - nxt
            F.flint_dense_gemv(x, Wgu, h, epilogue=F.FLINT_EPILOGUE_SWIGLU, flags=flags)
            F.flint_dense_gemv(h, Wdn, y[b % 2], flags=flags)
            y_prev = y[b % 2]
        for i, lay in enumerate(self.moe):
            yo = y[(N_DENSE + i) % 2]
            F.flint_moe_block(src, lay["router_w"], TOPK, lay["routed"], lay["shared"], ids[i], w[i], yo, self.ws,
                              y_prev=y_prev, residual_out=r[nxt], flags=flags, next=lay["next_pf"])
            src, nxt = r[nxt], 1 - nxt
            y_prev = yo
        F.flint_residual_rmsnorm(src, io["xf"], y_prev=y_prev, residual_out=io["r_final"], flags=flags)


def measure_stack(F, args, reps=20):
    """The full decode stack (49 blocks) per token step, PDL on and off, at
    T = 1 and (PDL on) T = 8, each step replayed from one CUDA graph."""
    import torch
    from nvfp4_moe_decode_sigmoid_gb300 import synth
    st = Stack("cuda")
    peak, _ = load_peaks()
    out = {}
    for T, pdl_modes in ((1, (True, False)), (8, (True,))):
        dev = "cuda"
        io = dict(x0=synth.activations(4242 + T, T, H, dev),
                  r=[torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)],
                  y=[torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)],
                  x=torch.empty((T, H), dtype=torch.bfloat16, device=dev),
                  h=torch.empty((T, DENSE_F), dtype=torch.bfloat16, device=dev),
                  xf=torch.empty((T, H), dtype=torch.bfloat16, device=dev),
                  r_final=torch.empty((T, H), dtype=torch.bfloat16, device=dev),
                  ids=[torch.empty((T, TOPK), dtype=torch.int32, device=dev) for _ in range(N_MOE)],
                  w=[torch.empty((T, TOPK), dtype=torch.float32, device=dev) for _ in range(N_MOE)])
        stream = torch.cuda.Stream()
        res = {}
        for pdl in pdl_modes:
            flags = F.FLINT_PDL if pdl else 0
            with torch.cuda.stream(stream):
                st.step(F, io, flags)  # warm-up; the routing of every block for the byte count
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    st.step(F, io, flags)
                for _ in range(3):
                    g.replay()
                stream.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            assert F.flint_workspace_check(st.ws) == F.FLINT_OK
            res[pdl] = e0.elapsed_time(e1) * 1e3 / reps
        distinct = [len(set(i.cpu().numpy().reshape(-1).tolist())) for i in io["ids"]]
        act = 2 * T * H * 2  # per block: residual + previous output in, new residual + output out (x, y)
        total = (N_DENSE * (st.dense_bytes() + act) + sum(step_bytes(d, T, False) + act for d in distinct)
                 + 2 * T * H * 2 * 2)
        us = res[True]
        ent = dict(us_per_step_pdl=round(us, 2), gb_s=round(total / (us * 1e-6) / 1e9, 1),
                   frac_of_peak=round(total / (us * 1e-6) / 1e9 / peak, 4), bytes_per_step=total,
                   mean_distinct_experts=round(sum(distinct) / len(distinct), 2),
                   launches_per_step=3 * N_DENSE + N_MOE + 1)
        if False in res:
            ent["us_per_step_no_pdl"] = round(res[False], 2)
        out[f"T{T}"] = ent
    del st
    torch.cuda.empty_cache()
    out["blocks"] = f"{N_DENSE} dense SwiGLU MLP ({H}->{DENSE_F}->{H}, NVFP4) + {N_MOE} MoE blocks, residual + RMSNorm"
    out["path"] = ("dense: flint_residual_rmsnorm -> flint_dense_gemv (SwiGLU) -> flint_dense_gemv; MoE: "
                   "flint_moe_block (norm fused, one cooperative kernel); final flint_residual_rmsnorm; one CUDA "
                   "graph per step")
    return out


PREFILL_T = 8192


def measure_prefill(F, reps=10):
    """The MoE layer over 8192 tokens (flint_moe_prefill: router GEMM, top-k,
    expert sort, grouped gate/up and down GEMMs on tcgen05, combine) on one
    full-size seeded layer; FLOPs = 2 x (router + 7 experts per token)."""
    import torch
    from nvfp4_moe_decode_sigmoid_gb300 import synth
    L = synth.Layer(1000, H=H, E=E, I=I, I_shared=I_SHARED, device="cuda")
    s = L.shared
    routed = F.Experts.from_gguf(L.gate, L.up, L.down, L.ts, E, H, I)
    shared = F.Experts.from_gguf(s["gate"], s["up"], s["down"], s["ts"].reshape(1, 3), 1, H, I_SHARED)
    T = PREFILL_T
    x = synth.activations(4242, T, H, "cuda")
    ws = torch.empty(F.flint_prefill_workspace_bytes(T, E, TOPK, H, I, I_SHARED), dtype=torch.uint8, device="cuda")
    F.flint_workspace_init(ws)
    ids = torch.empty((T, TOPK), dtype=torch.int32, device="cuda")
    w = torch.empty((T, TOPK), dtype=torch.float32, device="cuda")
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(3):
            F.flint_moe_prefill(x, L.router_w, TOPK, routed, shared, ids, w, y, ws)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            F.flint_moe_prefill(x, L.router_w, TOPK, routed, shared, ids, w, y, ws)
        e1.record(stream)
    torch.cuda.synchronize()
    assert F.flint_workspace_check(ws) == F.FLINT_OK
    us = e0.elapsed_time(e1) * 1e3 / reps
    flop = 2 * T * H * E + T * (TOPK + 1) * 2 * 3 * I * H
    peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        peak = 1900.0
    tf = flop / (us * 1e-6) / 1e12
    del L, s, routed, shared, ws
    torch.cuda.empty_cache()
    return dict(tokens=T, us=round(us, 1), tflops=round(tf, 1), flop=flop,
                roofline={"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
                          "frac": round(tf / peak, 4), "peak_note": "measured bf16 burst (cuBLAS)"},
                path="flint_moe_prefill: router GEMM, top-k, expert sort, grouped gate/up + down GEMMs "
                     "(tcgen05.mma kind::f16, NVFP4 dequantised to bf16 in shared memory), combine")


def measure_kernels(F, model, name, reps=8):
    """Average device duration of each kernel: the fused layer kernel, the
    router, flint_moe_decode as one kernel, and its gate/up and down kernels
    (the two-kernel path). For each, a CUDA graph of back-to-back
    launches (one per resident layer, no PDL) is replayed `reps` times between
    two CUDA events on the replay stream. The routing comes from a warm-up
    pass, so the gate/up and down launches see each layer's real selection."""
    import torch
    T, routing = WORKLOADS[name]
    nl = len(model.layers)
    bias, inp = make_inputs(model, T, routing, "cuda")
    for li in range(nl):
        run_step(F, model, inp, li, bias, 0, "chain")
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    calls = {
        "layer": lambda lay, io: F.flint_moe_layer(io["x"], lay["router_w"], TOPK, lay["routed"], lay["shared"],
                                                   io["ids"], io["w"], io["y"], model.ws, bias=bias,
                                                   next=lay["next_pf"]),
        "route": lambda lay, io: F.flint_moe_route(io["x"], lay["router_w"], TOPK, io["ids"], io["w"], model.ws,
                                                   bias=bias),
        "decode": lambda lay, io: F.flint_moe_decode(io["x"], io["ids"], io["w"], lay["routed"], lay["shared"],
                                                     io["y"], model.ws),
        "gate_up": lambda lay, io: F.flint_moe_gate_up(io["x"], io["ids"], lay["routed"], lay["shared"], model.ws),
        "down": lambda lay, io: F.flint_moe_down_combine(io["ids"], io["w"], lay["routed"], lay["shared"], io["y"],
                                                         model.ws),
    }
    out = {}
    for kname, call in calls.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for li in range(nl):
                    call(model.layers[li], inp[li])
            g.replay()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        assert F.flint_workspace_check(model.ws) == F.FLINT_OK, F.flint_last_error()
        out[kname + "_us"] = e0.elapsed_time(e1) * 1e3 / (reps * nl)
    gu_b, dn_b = expert_bytes()
    distinct = [len(set(io["ids"].cpu().numpy().reshape(-1).tolist())) for io in inp]
    out["gate_up_bytes"] = statistics.mean((d + 1) * (gu_b + 8) + T * H * 2 for d in distinct)
    out["down_bytes"] = statistics.mean((d + 1) * (dn_b + 4) + T * H * 2 for d in distinct)
    out["decode_bytes"] = out["gate_up_bytes"] + out["down_bytes"]
    out["route_bytes"] = ROUTER_BYTES + T * H * 2
    out["layer_bytes"] = statistics.mean(step_bytes(d, T, bias is not None) for d in distinct)
    return out


def measure_single_flushed(F, model, name, reps=7):
    """One flint_moe_layer call right after the L2 is flushed (a 512 MB write,
    four times the 129 MB L2), timed alone with CUDA events; median of `reps`."""
    import torch
    T, routing = WORKLOADS[name]
    bias, inp = make_inputs(model, T, routing, "cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    times = []
    with torch.cuda.stream(stream):
        for r in range(reps + 1):
            li = r % len(model.layers)
            flush.fill_(r & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run_step(F, model, inp, li, bias, 0, "fused")
            e1.record(stream)
            e1.synchronize()
            if r > 0:
                times.append(e0.elapsed_time(e1) * 1e3)
    assert F.flint_workspace_check(model.ws) == F.FLINT_OK, F.flint_last_error()
    del flush
    torch.cuda.empty_cache()
    return statistics.median(times)


def measure_e2e(F, model, name, steps, graph_steps):
    """Same metric through the C ABI with HOST buffers: every step moves its x
    from pinned host memory to the GPU and its y back, inside the timed region
    (a CUDA graph of R steps). Two ways are timed:
      copy:      cudaMemcpyAsync of x in, the layer on device buffers, y out;
      direct y:  x copied in, the layer writes y straight into the pinned host
                 buffer (GB300 reaches host memory coherently; with unified
                 addressing a pinned buffer has the same address on both sides;
                 each y row is written once), checked bit for bit against the
                 device-buffer result first.
    (Reading x from host memory inside the kernel as well measured 2.2x slower:
    every CTA reads all of x.) `value` is the faster of the two that passed."""
    import torch
    T, routing = WORKLOADS[name]
    nl = len(model.layers)
    bias, inp = make_inputs(model, T, routing, "cuda")
    hx = [io["x"].cpu().pin_memory() for io in inp]
    hy = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in inp]
    stream = torch.cuda.Stream()
    R = max(1, min(graph_steps, steps))
    reps = max(1, steps // R)

    def zero_copy_step(li, flags):
        lay, io = model.layers[li], inp[li]
        io["x"].copy_(hx[li], non_blocking=True)
        F.flint_moe_layer(io["x"], lay["router_w"], TOPK, lay["routed"], lay["shared"], io["ids"], io["w"], hy[li],
                          model.ws, bias=bias, flags=flags, next=lay["next_pf"])

    def copy_step(li, flags):
        inp[li]["x"].copy_(hx[li], non_blocking=True)
        run_step(F, model, inp, li, bias, flags, "fused")
        hy[li].copy_(inp[li]["y"], non_blocking=True)

    def timed(step):
        with torch.cuda.stream(stream):
            for s in range(nl):
                step(s % nl, F.FLINT_PDL)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for s in range(R):
                    step(s % nl, F.FLINT_PDL)
            g.replay()
            stream.synchronize()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1)

    def timed_overlapped():
        """x copies on a side stream of the same graph (each layer waits for its
        own copy's event, so the copy of step s + 1 overlaps step s); y written
        straight into pinned host memory by the layer."""
        side = torch.cuda.Stream()

        def capture_body():
            fork = torch.cuda.Event()
            fork.record(stream)
            side.wait_event(fork)
            evs = []
            with torch.cuda.stream(side):
                for s in range(R):
                    inp[s % nl]["x"].copy_(hx[s % nl], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(side)
                    evs.append(e)
            for s in range(R):
                li = s % nl
                stream.wait_event(evs[s])
                lay, io = model.layers[li], inp[li]
                F.flint_moe_layer(io["x"], lay["router_w"], TOPK, lay["routed"], lay["shared"], io["ids"], io["w"],
                                  hy[li], model.ws, bias=bias, flags=F.FLINT_PDL, next=lay["next_pf"])
        with torch.cuda.stream(stream):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                capture_body()
            g.replay()
            stream.synchronize()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1)

    # The graphs run steps 0..R-1, i.e. layers s % nl; only those layers' y
    # are written by the timed graph of every path (with R < nl the others
    # keep what an earlier pass left), so only those are compared.
    covered = sorted({s % nl for s in range(R)})

    def check_ws():
        assert F.flint_workspace_check(model.ws) == F.FLINT_OK, F.flint_last_error()

    ms_copy = timed(copy_step)
    check_ws()
    ref_y = [h.clone() for h in hy]          # y of every layer through device buffers
    same = lambda: all(torch.equal(hy[i].view(torch.int16), ref_y[i].view(torch.int16)) for i in covered)  # noqa: E731
    for h in hy:
        h.zero_()
    ms_zc = timed(zero_copy_step)
    check_ws()
    zc_ok = same()
    for h in hy:
        h.zero_()
    ms_ov = timed_overlapped()
    check_ws()
    ov_ok = same()
    distinct = [len(set(io["ids"].cpu().numpy().reshape(-1).tolist())) for io in inp]
    n = reps * R
    total = sum(step_bytes(distinct[s % nl], T, bias is not None) for s in range(R)) * reps
    paths = {"copy": (ms_copy, True, "pinned host x -> cudaMemcpyAsync -> flint_moe_layer -> cudaMemcpyAsync -> "
                                      "pinned host y, CUDA graph"),
             "direct_y": (ms_zc, zc_ok, "pinned host x -> cudaMemcpyAsync -> flint_moe_layer writing y into pinned "
                                        "host memory, CUDA graph"),
             "overlapped": (ms_ov, ov_ok, "pinned host x -> cudaMemcpyAsync on a side stream (step s + 1's copy "
                                          "overlaps step s) -> flint_moe_layer writing y into pinned host memory, one "
                                          "CUDA graph")}
    best = min((v[0], k) for k, v in paths.items() if v[1])[1]
    ms = paths[best][0]
    return dict(value=total / (ms * 1e-3) / 1e9, unit="GB/s", h2d_bytes_per_step=T * H * 2,
                d2h_bytes_per_step=T * H * 2, steps=n, us_per_step=ms * 1e3 / n, path=paths[best][2],
                us_per_step_by_path={k: round(v[0] * 1e3 / n, 3) for k, v in paths.items()},
                bit_identical_to_device_path={k: v[1] for k, v in paths.items()},
                layers_compared=len(covered))


def cpu_baseline(name, budget_s=20.0):
    """The oracle, as it stands, on this host, on a bounded sample of the same
    workload: whole layer steps (router + all selected experts + shared
    expert + combine) of the same recipe on a CPU-drawn layer. Two legs on
    the same inputs: the plain single-threaded build, and the same source
    built with OpenMP (output rows split over all host threads; the same
    bits). `value` is the OpenMP leg (the host's cores), when it exists."""
    import oracle
    from nvfp4_moe_decode_sigmoid_gb300 import synth
    T, routing = WORKLOADS[name]
    L = synth.Layer(1000, H=H, E=E, I=I, I_shared=I_SHARED, device="cpu")
    s = L.shared
    sh = dict(gate=s["gate"].numpy(), up=s["up"].numpy(), down=s["down"].numpy(), ts=s["ts"].numpy(), I=I_SHARED)
    bias = synth.zipf_bias(7, E).numpy() if routing == "zipf" else None
    wr = synth.bits(L.router_w)
    host_cores = os.cpu_count() or 1

    def leg(budget, max_steps):
        done, total_bytes, elapsed = 0, 0, 0.0
        outs = []
        while elapsed < budget and done < max_steps:
            x = synth.bits(synth.activations(5000 + done, T, H))
            t0 = time.perf_counter()
            ids, _, y = oracle.moe_layer(x, wr, TOPK, E, I, L.gate.numpy(), L.up.numpy(), L.down.numpy(),
                                         L.ts.numpy(), shared=sh, bias=bias)
            elapsed += time.perf_counter() - t0
            total_bytes += step_bytes(len(set(ids.reshape(-1).tolist())), T, bias is not None)
            outs.append(y)
            done += 1
        return total_bytes / elapsed / 1e9, done, elapsed, outs

    st_value, st_steps, st_s, st_out = leg(budget_s / 2, 64)
    out = dict(unit="GB/s", kind="oracle", host_cores=host_cores,
               single_thread={"value": st_value, "cores": 1, "steps": st_steps, "seconds": round(st_s, 2)})
    threads = oracle.use_openmp(0)
    try:
        if threads:
            mt_value, mt_steps, mt_s, mt_out = leg(budget_s / 2, 256)
            same = all(np.array_equal(a, b) for a, b in zip(st_out, mt_out))
            out.update(value=mt_value, cores=threads,
                       openmp={"value": mt_value, "cores": threads, "steps": mt_steps, "seconds": round(mt_s, 2),
                               "same_bits_as_single_thread": same},
                       sample=f"whole layer steps of {name} (T={T}) on a CPU-drawn layer: {mt_steps} steps in "
                              f"{mt_s:.1f} s on {threads} threads (OpenMP over output rows), {st_steps} steps in "
                              f"{st_s:.1f} s on one thread; host has {host_cores} cores")
        else:
            out.update(value=st_value, cores=1,
                       sample=f"{st_steps} whole layer steps of {name} (T={T}) on a CPU-drawn layer, {st_s:.1f} s, "
                              f"single thread (no OpenMP build on this host); host has {host_cores} cores")
    finally:
        oracle.use_openmp(-1)
    return out


def traffic_for(kernel_src_hash, tokens):
    """DRAM bytes per launch of the layer kernel that runs `tokens` tokens
    (the one-token kernel at one token, else the fused layer kernel) from the
    committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "layer_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("source_sha256") != kernel_src_hash:
        return None
    return (d.get("one_token") or {}).get("dram_bytes_per_launch") if tokens == 1 else d.get("dram_bytes_per_launch")


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for fn in ("layer.cu", "layer_one.cuh", "expert_common.cuh", "router_common.cuh", "flint_device.cuh",
               "flint_internal.h"):
        with open(os.path.join(ROOT, "nvfp4_moe_decode_sigmoid_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def run_flint(args):
    import torch
    import torch.distributed as dist
    from nvfp4_moe_decode_sigmoid_gb300 import _build
    _build.build()
    from nvfp4_moe_decode_sigmoid_gb300 import flint as F

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def sync_all():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v):
        return replica_max(v, world, "cuda")

    model = Model(args.layers, "cuda")
    dev_index = torch.cuda.current_device()
    main = measure_workload(F, model, args.workload, args.steps, args.warmup, args.graph_steps, sync_all, dev_index)
    ms = max_over_ranks(main["ms"])
    value = replica_value(main["bytes"], world, ms)
    chain = measure_workload(F, model, args.workload, max(1024, args.steps // 4), args.warmup, args.graph_steps,
                             sync_all, dev_index, with_clocks=False, path="chain")
    chain3 = measure_workload(F, model, args.workload, max(1024, args.steps // 4), args.warmup, args.graph_steps,
                              sync_all, dev_index, with_clocks=False, path="chain3")
    extra = {}
    if not args.no_extra:
        for name in WORKLOADS:
            if name == args.workload:
                continue
            r = measure_workload(F, model, name, max(1024, args.steps // 4), args.warmup, args.graph_steps, sync_all,
                                 dev_index, with_clocks=False)
            extra[name] = dict(us_per_layer=r["ms"] * 1e3 / r["steps"], gb_s=r["bytes"] / (r["ms"] * 1e-3) / 1e9,
                               mean_distinct_experts=r["mean_distinct"], bytes_per_step=r["bytes_per_step_mean"])
    kern = measure_kernels(F, model, args.workload)
    kern["single_call_l2_flushed_us"] = measure_single_flushed(F, model, args.workload)
    bf16 = {}
    if not args.no_bf16:
        bf16 = measure_bf16(F, model, args, sync_all, dev_index)

    peak, peak_src = load_peaks()
    achieved = kern["layer_bytes"] / (kern["layer_us"] * 1e-6) / 1e9
    traffic = traffic_for(kernel_source_hash(), WORKLOADS[args.workload][0])
    e2e = measure_e2e(F, model, args.workload, min(args.steps, 8192), args.graph_steps)
    stack, prefill = {}, {}
    if not args.no_stack or not args.no_prefill:
        del model
        torch.cuda.empty_cache()
    if not args.no_stack:
        stack = measure_stack(F, args)
    if not args.no_prefill:
        prefill = measure_prefill(F)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload)
    T, routing = WORKLOADS[args.workload]
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms / args.steps,
            "us_per_layer": ms * 1e3 / args.steps,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": args.workload, "tokens": T, "routing": routing, "hidden": H, "experts": E,
                       "top_k": TOPK, "inter": I, "shared_inter": I_SHARED, "weights": "nvfp4 (e2m1 + ue4m3/16 + fp32)",
                       "activations": "bf16", "layers_rotated": args.layers, "pdl": True,
                       "prefetch": "each layer pulls the next one's router and shared expert into L2 before its "
                                   "PDL wait",
                       "path": "flint_moe_layer: one cooperative kernel per layer",
                       "graph_steps": args.graph_steps,
                       "l2": f"inputs larger than L2: {args.layers} resident layers cycled, reuse distance "
                             f"{(args.layers - 1) * main['bytes_per_step_mean'] / 1e6:.0f} MB > 129 MB L2",
                       "parallelism": f"replicas x{world}",
                       "mean_distinct_experts": main["mean_distinct"],
                       "bytes_per_step": main["bytes_per_step_mean"]},
            "roofline": {"bound": "hbm", "kernel": "layer_one_kernel" if T == 1 else "layer_kernel",
                         "achieved": round(achieved, 1),
                         "peak": peak, "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                         "traffic": traffic, "algorithmic_bytes_per_launch": kern["layer_bytes"],
                         "us_per_launch": kern["layer_us"]},
            "kernels_us": {k: round(v, 3) for k, v in kern.items() if k.endswith("_us")},
            "kernels_gb_s": {k: round(kern[k + "_bytes"] / (kern[k + "_us"] * 1e-6) / 1e9, 1)
                             for k in ("layer", "route", "decode", "gate_up", "down")},
            "route_decode_chain": {"us_per_layer": round(chain["ms"] * 1e3 / chain["steps"], 3),
                                   "gb_s": round(chain["bytes"] / (chain["ms"] * 1e-3) / 1e9, 1),
                                   "path": "flint_moe_route -> flint_moe_decode (one cooperative kernel, routing "
                                           "given), PDL"},
            "three_kernel_chain": {"us_per_layer": round(chain3["ms"] * 1e3 / chain3["steps"], 3),
                                   "gb_s": round(chain3["bytes"] / (chain3["ms"] * 1e-3) / 1e9, 1),
                                   "path": "flint_moe_route -> flint_moe_decode on a workspace sized without the "
                                           "hidden size (gate/up, down), PDL"},
            "layer_frac_of_peak": round(value / world / peak, 4),
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": main["clocks"],
            "extra_workloads": extra,
            "bf16_experts": bf16,
            "decode_stack": stack,
            "prefill": prefill,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the oracle, on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on this host's cores
    (the OpenMP build over output rows where the compiler has OpenMP, else
    the plain build on one thread), on the workload this bench is labelled
    with. A step is the whole layer for the workload's T tokens (router, the
    selected experts, the shared expert, combine), with fresh x per step.
    Where K + W whole steps would not end within the time budget, each step
    is a bounded sample instead: a slice of gate rows of one selected expert
    (the GEMVs carry 92% of the layer's bytes), said so in `sample`."""
    rank, world, local = dist_env()
    if rank != 0:
        return
    import oracle
    from nvfp4_moe_decode_sigmoid_gb300 import synth
    T, routing = WORKLOADS[args.workload]
    L = synth.Layer(1000, H=H, E=E, I=I, I_shared=I_SHARED, device="cpu")
    s = L.shared
    sh = dict(gate=s["gate"].numpy(), up=s["up"].numpy(), down=s["down"].numpy(), ts=s["ts"].numpy(), I=I_SHARED)
    bias = synth.zipf_bias(7, E).numpy() if routing == "zipf" else None
    wr = synth.bits(L.router_w)
    host_cores = os.cpu_count() or 1
    threads = oracle.use_openmp(0) or 1
    budget = 150.0
    total = args.steps + args.warmup
    per_step = budget / max(total, 1)
    gu_bytes_row = H // 64 * 36  # GGUF and kernel layouts both hold 0.5625 B per weight

    def whole_step(seed):
        x = synth.bits(synth.activations(seed, T, H))
        t0 = time.perf_counter()
        ids, _, _ = oracle.moe_layer(x, wr, TOPK, E, I, L.gate.numpy(), L.up.numpy(), L.down.numpy(), L.ts.numpy(),
                                     shared=sh, bias=bias)
        return time.perf_counter() - t0, step_bytes(len(set(ids.reshape(-1).tolist())), T, bias is not None), ids

    t_step, _, ids1 = whole_step(9000)
    whole = t_step <= per_step
    gate_np = L.gate.numpy()
    sel = sorted({int(e) for e in ids1.reshape(-1)})
    x1 = synth.bits(synth.activations(9000, 1, H))
    rows_per_step = 0
    if not whole:
        rows_per_step = min(I, max(1, int(I * len(sel) * per_step / max(t_step, 1e-9) / 2)))
    timed_s, timed_b, cursor = 0.0, 0, 0
    for i in range(total):
        if whole:
            t, b, _ = whole_step(9001 + i)
        else:
            e = sel[cursor % len(sel)]
            cursor += 1
            W = gate_np[e][: rows_per_step * gu_bytes_row]
            t0 = time.perf_counter()
            oracle.dense_gemv(x1, W, rows_per_step, ts=(float(L.ts[e, 0]),))
            t = time.perf_counter() - t0
            b = rows_per_step * gu_bytes_row
        if i >= args.warmup:
            timed_s += t
            timed_b += b
    oracle.use_openmp(-1)
    value = timed_b / max(timed_s, 1e-12) / 1e9
    how = f"{threads} threads (OpenMP over output rows)" if threads > 1 else "one thread"
    sample = (f"whole layer steps of {args.workload}: {T} tokens per step through the router, the selected "
              f"experts, the shared expert and the combine, {how}, host has {host_cores} cores"
              if whole else
              f"{rows_per_step} gate rows of one selected expert per step (oracle expert GEMV), cycling over the "
              f"{len(sel)} experts the workload's tokens select, {how}, host has {host_cores} cores")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": timed_s * 1e3 / max(args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload, "tokens": T, "routing": routing, "whole_layer_steps": whole},
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": threads, "host_cores": host_cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.prefill_only:
        import torch
        from nvfp4_moe_decode_sigmoid_gb300 import _build
        _build.build()
        from nvfp4_moe_decode_sigmoid_gb300 import flint as F
        torch.cuda.set_device(dist_env()[2])
        r = measure_prefill(F)
        print(json.dumps({"metric": "MoE-layer prefill TFLOP/s (8192 tokens)", "value": r["tflops"],
                          "unit": "TFLOP/s", "higher_is_better": True, "prefill": r}), flush=True)
    else:
        run_flint(args)


if __name__ == "__main__":
    main()
