"""GPU repack, unrepack and dequant against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from flint_testlib import flint
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,rows,cols", [(1, 1, 64), (3, 5, 192), (2, 16, 256), (4, 33, 2048), (2, 2048, 512),
                                         (1, 7, 6144)])
def test_repack_matches_oracle_bytes(n, rows, cols):
    f = flint()
    src = synth.gguf_nvfp4(100 + rows + cols, n, rows, cols)
    dst = torch.full((f.flint_nvfp4_packed_bytes(n, rows, cols),), 0xAB, dtype=torch.uint8, device="cuda")
    f.flint_nvfp4_repack(src.cuda(), n, rows, cols, dst)
    torch.cuda.synchronize()
    ref = oracle.repack(src.numpy().reshape(-1), n, rows, cols)
    assert np.array_equal(dst.cpu().numpy(), ref)
    back = torch.zeros(src.numel(), dtype=torch.uint8, device="cuda")
    f.flint_nvfp4_unrepack(dst, n, rows, cols, back)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), src.numpy().reshape(-1))


def test_repack_into_gate_up_layout_with_stride():
    f = flint()
    E, I, H = 3, 256, 1024
    gate = synth.gguf_nvfp4(1, E, I, H)
    up = synth.gguf_nvfp4(2, E, I, H)
    rs = f.flint_nvfp4_row_stride(H)
    gu = torch.zeros(E * 2 * I * rs, dtype=torch.uint8, device="cuda")
    f.flint_nvfp4_repack(gate.cuda(), E, I, H, gu, 2 * I * rs, 0)
    f.flint_nvfp4_repack(up.cuda(), E, I, H, gu, 2 * I * rs, I * rs)
    torch.cuda.synchronize()
    got = gu.cpu().numpy().reshape(E, 2, I * rs)
    assert np.array_equal(got[:, 0].reshape(-1), oracle.repack(gate.numpy().reshape(-1), E, I, H))
    assert np.array_equal(got[:, 1].reshape(-1), oracle.repack(up.numpy().reshape(-1), E, I, H))


def test_exhaustive_scale_bytes_and_codes_round_trip():
    f = flint()
    rows, cols = 256, 64
    rng = np.random.default_rng(7)
    src = rng.integers(0, 256, (rows, 36), dtype=np.uint8)
    src[:, :4] = np.arange(256, dtype=np.uint8)[:, None]
    src[:16, 4:] = np.arange(16, dtype=np.uint8)[:, None] * 0x11
    s = torch.from_numpy(src.reshape(-1)).cuda()
    dst = torch.empty(f.flint_nvfp4_packed_bytes(1, rows, cols), dtype=torch.uint8, device="cuda")
    f.flint_nvfp4_repack(s, 1, rows, cols, dst)
    back = torch.empty_like(s)
    f.flint_nvfp4_unrepack(dst, 1, rows, cols, back)
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy(), oracle.repack(src.reshape(-1), 1, rows, cols))
    assert np.array_equal(back.cpu().numpy(), src.reshape(-1))


@pytest.mark.parametrize("rows,cols", [(3, 64), (64, 512), (8, 2048)])
def test_dequant_is_bit_exact(rows, cols):
    f = flint()
    src = synth.gguf_nvfp4(9 + rows, 1, rows, cols)
    dst = torch.empty(f.flint_nvfp4_packed_bytes(1, rows, cols), dtype=torch.uint8, device="cuda")
    f.flint_nvfp4_repack(src.cuda(), 1, rows, cols, dst)
    out = torch.empty(rows * cols, dtype=torch.float32, device="cuda")
    f.flint_nvfp4_dequant(dst, rows, cols, out)
    torch.cuda.synchronize()
    ref = oracle.gguf_decode(src.numpy().reshape(-1), rows, cols).reshape(-1)
    got = out.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_dequant_every_code_and_scale():
    # all 16 codes under every UE4M3 scale byte 0x00..0x7E (0x7F is NaN, outside the domain)
    f = flint()
    rows, cols = 127, 64
    src = np.zeros((rows, 36), np.uint8)
    src[:, :4] = np.arange(127, dtype=np.uint8)[:, None]
    src[:, 4:] = np.tile(np.array([0x80, 0x91, 0xA2, 0xB3, 0xC4, 0xD5, 0xE6, 0xF7], np.uint8), 4)
    dst = torch.empty(f.flint_nvfp4_packed_bytes(1, rows, cols), dtype=torch.uint8, device="cuda")
    f.flint_nvfp4_repack(torch.from_numpy(src.reshape(-1)).cuda(), 1, rows, cols, dst)
    out = torch.empty(rows * cols, dtype=torch.float32, device="cuda")
    f.flint_nvfp4_dequant(dst, rows, cols, out)
    torch.cuda.synchronize()
    ref = oracle.gguf_decode(src.reshape(-1), rows, cols).reshape(-1)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), ref)


def test_empty_repack_is_a_no_op():
    f = flint()
    d = torch.zeros(16, dtype=torch.uint8, device="cuda")
    f.flint_nvfp4_repack(d, 0, 4, 64, d)
    f.flint_nvfp4_repack(d, 2, 0, 64, d)
    torch.cuda.synchronize()
    assert not d.any()
