"""Oracle self-tests: number formats and the NVFP4 repack (CPU only).

Pins: a hand-decoded E2M1 table, torch's float8_e4m3fn for UE4M3, torch's
bf16 rounding, a hand-derived GGUF superblock and its hand-derived kernel
layout, and the repack round trip.
"""
import numpy as np
import pytest
import torch

import oracle
from golden_io import read_fixture
from nvfp4_moe_decode_sigmoid_gb300 import synth

# E2M1 (OCP FP4) decoded by hand: codes 0..7 positive, 8..15 their negatives.
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_hand_table():
    got = [oracle.e2m1_value(c) for c in range(16)]
    assert got == E2M1_TABLE
    assert np.signbit(oracle.e2m1_value(8))  # code 8 is -0


def test_ue4m3_matches_library_e4m3():
    # positive E4M3 (bit 7 clear) is UE4M3; torch's float8_e4m3fn is an
    # independent implementation of the same bit layout.
    b = torch.arange(0, 0x7F, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.ue4m3_value(int(v)) for v in range(0x7F)])
    assert np.array_equal(got, ref)
    assert np.isnan(oracle.ue4m3_value(0x7F))


def test_ue4m3_landmarks_and_bit7():
    assert oracle.ue4m3_value(0x01) == 2.0 ** -9  # smallest subnormal
    assert oracle.ue4m3_value(0x08) == 2.0 ** -6  # smallest normal
    assert oracle.ue4m3_value(0x38) == 1.0
    assert oracle.ue4m3_value(0x7E) == 448.0      # largest finite
    for v in range(0x7F):
        assert oracle.ue4m3_value(v | 0x80) == oracle.ue4m3_value(v)


def test_bf16_round_matches_library_on_floats():
    rng = np.random.default_rng(5)
    parts = [
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormal range
        (rng.standard_normal(2000) * 3e38).astype(np.float32),    # near overflow
        np.array([0.0, -0.0, 1.0, 3.3895314e38, 3.4e38, 1e-45, -1e-45], np.float32),
    ]
    # exact ties: bf16 values plus half an ulp
    base = rng.integers(0, 0x7F00, 4000, dtype=np.uint32) << 16
    parts.append((base | 0x8000).view(np.float32))
    f = np.concatenate(parts)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(f.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_round_is_nearest_for_doubles():
    # doubles that fall between floats: the result must be the nearest bf16
    rng = np.random.default_rng(6)
    v = rng.standard_normal(3000) * np.exp2(rng.integers(-60, 60, 3000))
    got = oracle.bf16_round(v)
    vals = oracle.bf16_value(got)
    up = oracle.bf16_value((got.astype(np.int32) + 1).astype(np.uint16))
    dn = oracle.bf16_value((got.astype(np.int32) - 1).astype(np.uint16))
    err = np.abs(vals - v)
    assert np.all(err <= np.abs(up - v)) and np.all(err <= np.abs(dn - v))


def test_bf16_value_round_trip_all_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_value(pats)
    finite = np.isfinite(vals)
    back = oracle.bf16_round(vals[finite])
    assert np.array_equal(back, pats[finite])


def test_gguf_superblock_fixture():
    fx = read_fixture("nvfp4_superblock.txt")
    got = oracle.gguf_decode(fx["bytes"], 1, 64)[0]
    assert np.array_equal(got, fx["values"])
    assert np.array_equal(np.signbit(got), np.signbit(fx["values"]))  # -0 where the codes say so


def test_kernel_layout_fixture():
    sb = read_fixture("nvfp4_superblock.txt")["bytes"]
    fx = read_fixture("kernel_layout_1x64.txt")
    assert oracle.packed_row_stride(64) == fx["row_stride"]
    assert np.array_equal(oracle.repack(sb, 1, 1, 64), fx["bytes"])
    assert np.array_equal(oracle.packed_decode(fx["bytes"], 1, 64)[0],
                          read_fixture("nvfp4_superblock.txt")["values"])


@pytest.mark.parametrize("rows,cols,n", [(3, 64, 2), (5, 192, 1), (16, 256, 3), (4, 2048, 1)])
def test_repack_round_trip_and_values(rows, cols, n):
    src = synth.gguf_nvfp4(11 + rows, n, rows, cols).numpy().reshape(-1)
    dst = oracle.repack(src, n, rows, cols)
    assert np.array_equal(oracle.unrepack(dst, n, rows, cols), src)
    per = oracle.gguf_matrix_bytes(rows, cols)
    ms = rows * oracle.packed_row_stride(cols)
    for m in range(n):
        a = oracle.gguf_decode(src[m * per:(m + 1) * per], rows, cols)
        b = oracle.packed_decode(dst[m * ms:(m + 1) * ms], rows, cols)
        assert np.array_equal(a, b, equal_nan=True)


def test_repack_exhaustive_scale_bytes_and_codes():
    # every scale byte value (bit 7 included) and every code in every nibble slot
    rows, cols = 256, 64
    rng = np.random.default_rng(7)
    src = rng.integers(0, 256, (rows, 36), dtype=np.uint8)
    src[:, :4] = np.arange(256, dtype=np.uint8)[:, None]
    src[:16, 4:] = (np.arange(16, dtype=np.uint8)[:, None] * 0x11)
    src = src.reshape(-1)
    dst = oracle.repack(src, 1, rows, cols)
    assert np.array_equal(oracle.unrepack(dst, 1, rows, cols), src)


def test_repack_with_matrix_stride_leaves_gaps():
    rows, cols, n = 4, 128, 3
    src = synth.gguf_nvfp4(3, n, rows, cols).numpy().reshape(-1)
    rs = oracle.packed_row_stride(cols)
    ms = 2 * rows * rs  # e.g. gate rows of a [2I, H] gate/up matrix
    dst = oracle.repack(src, n, rows, cols, dst_mat_stride=ms)
    for m in range(n):
        assert not dst[m * ms + rows * rs:(m + 1) * ms].any()
    assert np.array_equal(oracle.unrepack(dst, n, rows, cols, dst_mat_stride=ms), src)
