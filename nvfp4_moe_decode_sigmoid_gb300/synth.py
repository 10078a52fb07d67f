"""Seeded synthetic inputs for the MoE decode step.

This module only draws random numbers in the shapes, formats and
distributions of the workloads; it holds none of the method's arithmetic.
The CUDA path, the oracle, the tests and the benchmark all take their inputs
from here.

Recipe (one Flint-style MoE layer; hidden size H = 2048, E = 256 routed
experts, k = 6, intermediate size I = 512 for routed and shared experts):

* NVFP4 weights are GGUF superblocks of 36 bytes per 64 values: bytes 0..3
  are UE4M3 block scales with exponent field uniform in 1..7 and mantissa
  uniform in 0..7 (values 2^-6 .. 1.875), bytes 4..35 are E2M1 codes, every
  nibble uniform over its 16 values.
* One FP32 tensor scale per (expert, matrix), uniform in [0.02, 0.06].
* Activations x ~ N(0, 1), each token scaled to unit RMS, stored as bf16.
* Router weights bf16 ~ N(0, 0.02^2), shape [E, H].
* BF16 expert weights (the 16-bit checkpoint variant) ~ N(0, 0.02^2).
* Skewed routing: a seeded permutation gives expert e a rank r_e in 1..E and
  the router bias is ln(r_e^-1.1 / sum_r r^-1.1) (a Zipf(1.1) prior).

Every generator takes an explicit seed; the same seed gives the same bytes
on every platform (torch's CPU generator). On a CUDA device the same recipe is
drawn from torch's CUDA generator instead (different bytes, same
distribution), which is how the benchmark fills gigabytes of resident layers
quickly.
"""
from __future__ import annotations

import math

import torch

SB_VALUES = 64
SB_BYTES = 36


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _mix(*parts: int) -> int:
    """Derive a sub-seed from integers (a fixed polynomial hash)."""
    h = 1469598103934665603
    for p in parts:
        h = ((h ^ (int(p) & 0xFFFFFFFFFFFF)) * 1099511628211) & 0x7FFF_FFFF_FFFF_FFFF
    return h


def gguf_nvfp4(seed: int, n_mats: int, rows: int, cols: int, device="cpu") -> torch.Tensor:
    """Random GGUF NVFP4 matrices: uint8 [n_mats, rows * cols/64 * 36]."""
    assert cols % SB_VALUES == 0
    g = _gen(seed, device)
    nsb = n_mats * rows * (cols // SB_VALUES)
    blk = torch.randint(0, 256, (nsb, SB_BYTES), generator=g, device=device, dtype=torch.uint8)
    e = torch.randint(1, 8, (nsb, 4), generator=g, device=device, dtype=torch.uint8)
    m = torch.randint(0, 8, (nsb, 4), generator=g, device=device, dtype=torch.uint8)
    blk[:, :4] = (e << 3) | m
    return blk.reshape(n_mats, -1)


def tensor_scales(seed: int, shape, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return (0.02 + 0.04 * torch.rand(shape, generator=g, device=device, dtype=torch.float32)).contiguous()


def bf16_normal(seed: int, shape, std: float, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def activations(seed: int, T: int, H: int, device="cpu") -> torch.Tensor:
    """x ~ N(0,1) per element, each row scaled to unit RMS, bf16 [T, H]."""
    g = _gen(seed, device)
    x = torch.randn((T, H), generator=g, device=device, dtype=torch.float32)
    x = x / x.pow(2).mean(dim=1, keepdim=True).sqrt()
    return x.to(torch.bfloat16)


def zipf_bias(seed: int, E: int, s: float = 1.1) -> torch.Tensor:
    """Router bias of a Zipf(s) prior over a seeded ranking of the experts."""
    g = _gen(seed, "cpu")
    ranks = torch.randperm(E, generator=g) + 1
    norm = sum(r ** -s for r in range(1, E + 1))
    return torch.tensor([math.log(int(r) ** -s / norm) for r in ranks], dtype=torch.float32)


def bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit pattern (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


class Layer:
    """Seeded weights of one MoE layer, drawn on `device`.

    nvfp4: gate/up [E, I*H/64*36] and down [E, H*I/64*36] GGUF bytes,
           ts [E, 3] (gate, up, down); the shared expert likewise with E = 1.
    bf16:  gate/up [E, I, H], down [E, H, I] bf16 tensors; no tensor scales.
    """

    def __init__(self, seed: int, H: int = 2048, E: int = 256, I: int = 512, I_shared: int = 512,
                 wdtype: str = "nvfp4", device="cpu", shared: bool = True):
        self.seed, self.H, self.E, self.I, self.Is = seed, H, E, I, I_shared
        self.wdtype, self.device = wdtype, device
        s = lambda kind: _mix(seed, kind)  # noqa: E731
        self.router_w = bf16_normal(s(1), (E, H), 0.02, device)
        if wdtype == "nvfp4":
            self.gate = gguf_nvfp4(s(2), E, I, H, device)
            self.up = gguf_nvfp4(s(3), E, I, H, device)
            self.down = gguf_nvfp4(s(4), E, H, I, device)
            self.ts = tensor_scales(s(5), (E, 3), device)
        else:
            self.gate = bf16_normal(s(2), (E, I, H), 0.02, device)
            self.up = bf16_normal(s(3), (E, I, H), 0.02, device)
            self.down = bf16_normal(s(4), (E, H, I), 0.02, device)
            self.ts = None
        self.shared = None
        if shared and I_shared > 0:
            if wdtype == "nvfp4":
                self.shared = dict(gate=gguf_nvfp4(s(6), 1, I_shared, H, device),
                                   up=gguf_nvfp4(s(7), 1, I_shared, H, device),
                                   down=gguf_nvfp4(s(8), 1, H, I_shared, device),
                                   ts=tensor_scales(s(9), (3,), device), I=I_shared)
            else:
                self.shared = dict(gate=bf16_normal(s(6), (1, I_shared, H), 0.02, device),
                                   up=bf16_normal(s(7), (1, I_shared, H), 0.02, device),
                                   down=bf16_normal(s(8), (1, H, I_shared), 0.02, device),
                                   ts=None, I=I_shared)

    def x(self, T: int, rep: int = 0) -> torch.Tensor:
        return activations(_mix(self.seed, 100, rep), T, self.H, self.device)
