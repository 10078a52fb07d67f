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


@pytest.mark.parametrize("T,lost", [(2, "cta0"), (1, "cta0"), (1, "router_row")])
def test_fused_layer_lost_cta_times_out_and_the_workspace_recovers(T, lost):
    """The fused layer with one CTA that publishes no router scores (the test
    hook): the others' bounded waits run out after the short budget, the call
    records FLINT_ERR_TIMEOUT, and flint_workspace_check re-initialises the
    workspace. A later call on the same workspace is correct again (oracle),
    and one made before the check does nothing and keeps the error. At one
    token (the one-token kernel: E = 16 router rows spread over all CTAs) the
    lost CTA is CTA 0, which holds no router row and withholds its h count,
    or the first CTA that holds a router row."""
    import numpy as np

    import oracle
    from flint_testlib import DeviceLayer, assert_close, combine_terms, margin_x

    f = flint()
    dl = DeviceLayer(synth.Layer(17, H=1024, E=16, I=256, I_shared=256))
    k, H = 6, 1024
    x = margin_x(synth.bits(dl.L.router_w), T, H, k, None, seed=3)
    ws = dl.workspace(k)
    ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    y = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    xc = x.cuda()

    def call():
        f.flint_moe_layer(xc, dl.router_w, k, dl.routed, dl.shared, ids, w, y, ws)

    f.flint_workspace_set_wait_budget(ws, 2000)  # 2 ms
    G = torch.cuda.get_device_properties(0).multi_processor_count
    cta = 0 if lost == "cta0" else next(c for c in range(G) if (c + 1) * 16 // G > c * 16 // G)
    f.flint_selftest_lose_cta(ws, cta)           # this CTA publishes nothing
    call()
    torch.cuda.synchronize()
    call()                                       # before the check: returns at once
    torch.cuda.synchronize()
    assert f.flint_workspace_check(ws) == f.FLINT_ERR_TIMEOUT
    assert f.flint_workspace_check(ws) == f.FLINT_OK  # re-initialised: hook and status gone
    y.zero_()
    call()
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    rids, rw, ry = oracle.moe_layer(synth.bits(x), synth.bits(dl.L.router_w), k, **dl.oracle_args())
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert_close(synth.bits(y), ry, "after recovery", terms=combine_terms(synth.bits(x), rids, rw, dl))


@pytest.mark.parametrize("T", [1, 2])
def test_decode_one_kernel_lost_cta_times_out_and_the_workspace_recovers(T):
    """flint_moe_decode on a workspace sized for one kernel, with CTA 0 (a
    shared-expert CTA) publishing no h counts: the CTAs that wait for them give
    up after the short budget, the check reports FLINT_ERR_TIMEOUT and
    re-initialises the workspace, and the next call is correct (oracle)."""
    import numpy as np

    import oracle
    from flint_testlib import DeviceLayer, assert_close, combine_terms

    f = flint()
    dl = DeviceLayer(synth.Layer(19, H=1024, E=16, I=256, I_shared=256))
    k, H = 4, 1024
    ids = np.array([[2, 9, 4, 11], [0, 9, 15, 6]][:T], np.int32)
    w = np.array([[0.4, 0.3, 0.2, 0.1], [0.1, 0.2, 0.3, 0.4]][:T], np.float32)
    x = synth.activations(5 + T, T, H)
    ws = dl.workspace(k)
    y = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    xc, ic, wc = x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()

    def call():
        f.flint_moe_decode(xc, ic, wc, dl.routed, dl.shared, y, ws)

    f.flint_workspace_set_wait_budget(ws, 2000)  # 2 ms
    f.flint_selftest_lose_cta(ws, 0)
    call()
    torch.cuda.synchronize()
    assert f.flint_workspace_check(ws) == f.FLINT_ERR_TIMEOUT
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    call()
    assert f.flint_workspace_check(ws) == f.FLINT_OK
    ref = oracle.moe_experts(synth.bits(x), ids, w, **dl.oracle_args())
    assert_close(synth.bits(y), ref, "after recovery", terms=combine_terms(synth.bits(x), ids, w, dl))
