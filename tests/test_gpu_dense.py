"""GPU dense GEMV on packed NVFP4 weights (plain and SwiGLU epilogue) against
the oracle."""
import pytest
import torch

import oracle
from flint_testlib import assert_close, flint
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K,T", [(2048, 6144, 1), (2048, 6144, 8), (300, 1024, 3), (64, 1024, 2), (4096, 2048, 5), (100, 3072, 7)])
def test_dense_plain(N, K, T):
    f = flint()
    src = synth.gguf_nvfp4(N + K, 1, N, K)
    ts = torch.tensor([0.04], dtype=torch.float32)
    W = f.Packed.from_gguf(src.cuda(), N, K, ts)
    x = synth.activations(N + T, T, K)
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    f.flint_dense_gemv(x.cuda(), W, y)
    torch.cuda.synchronize()
    ref = oracle.dense_gemv(synth.bits(x), src.numpy().reshape(-1), N, ts=(0.04,))
    assert_close(synth.bits(y), ref, "dense")


@pytest.mark.parametrize("N,K,T", [(12288, 2048, 1), (12288, 2048, 8), (512, 1024, 3)])
def test_dense_swiglu(N, K, T):
    f = flint()
    src = synth.gguf_nvfp4(N * 3 + K, 1, N, K)
    ts = torch.tensor([0.03, 0.05], dtype=torch.float32)
    W = f.Packed.from_gguf(src.cuda(), N, K, ts)
    x = synth.activations(N + T + 1, T, K)
    y = torch.empty((T, N // 2), dtype=torch.bfloat16, device="cuda")
    f.flint_dense_gemv(x.cuda(), W, y, epilogue=f.FLINT_EPILOGUE_SWIGLU)
    torch.cuda.synchronize()
    ref = oracle.dense_gemv(synth.bits(x), src.numpy().reshape(-1), N, ts=(0.03, 0.05), epilogue=oracle.EPI_SWIGLU)
    assert_close(synth.bits(y), ref, "dense swiglu")
