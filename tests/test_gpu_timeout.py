"""A bounded device wait that nothing completes gives up, records a timeout in
the workspace status word, and leaves the context usable."""
import pytest
import torch

from flint_testlib import flint
from nvfp4_moe_decode_sigmoid_gb300 import synth

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    f = flint()
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    f.flint_workspace_init(ws)
    f.flint_selftest_wait_timeout(ws, 20_000_000)  # 20 ms
    assert f.flint_workspace_check(ws) == f.FLINT_ERR_TIMEOUT
    assert f.flint_workspace_check(ws) == f.FLINT_OK  # status cleared
    # the context still works: run a real kernel afterwards
    src = synth.gguf_nvfp4(1, 1, 4, 64).cuda()
    dst = torch.empty(f.flint_nvfp4_packed_bytes(1, 4, 64), dtype=torch.uint8, device="cuda")
    f.flint_nvfp4_repack(src, 1, 4, 64, dst)
    torch.cuda.synchronize()
