"""The phase-trace tool's report of the one-token kernel on synthetic stamps
(no GPU): every interval is the median / max of the stamp differences over
the CTAs of the calls traced, the decode path drops the router's intervals,
and consecutive calls give the gap between them."""
import argparse

import numpy as np

from nvfp4_moe_decode_sigmoid_gb300 import phase_trace as pt


def _trace(calls=4, ctas=8):
    """Stamps of `calls` calls of `ctas` CTAs: stamp i at 1000 * i cycles plus
    the CTA index (so every interval is 1000 * (b - a) cycles), role byte 2, the
    global timer entry at 10 us per call and end 8 us after it."""
    tr = np.zeros((pt.N_CALLS, pt.N_CTAS, pt.N_STAMPS), np.int64)
    for c in range(calls):
        for k in range(ctas):
            for i in range(15):
                tr[c, k, i] = 1000 * i + k + 1
            tr[c, k, 3] = 1000 * 3 + k + 1
            tr[c, k, 26] = 1
            tr[c, k, 28] = 2
            tr[c, k, 29] = 10_000 * c + 100 * k
            tr[c, k, 30] = 10_000 * c + 8_000
            tr[c, k, 31] = c + 1
    return tr[:, :ctas], list(range(calls))


def test_one_token_report_intervals_and_call_gap(capsys):
    tr, calls = _trace()
    pt.report_one(argparse.Namespace(routing="uniform", layers=32, path="layer"), tr, calls, tr.shape[1])
    out = capsys.readouterr().out
    rows = {line.split(" | ")[0].strip("| "): line for line in out.splitlines() if line.startswith("| ")}
    for name, a, b in pt.INTERVALS_ONE:
        assert name in rows, name
        assert rows[name].endswith(f"| {(b - a):.2f} / {(b - a):.2f} |"), rows[name]
    # the next call's first entry is 10 - 8 = 2 us after this call's end
    assert "first entry of the next call minus last end of this one 2.00 us" in out


def test_decode_path_drops_the_router_intervals(capsys):
    tr, calls = _trace()
    pt.report_one(argparse.Namespace(routing="uniform", layers=32, path="decode"), tr, calls, tr.shape[1])
    out = capsys.readouterr().out
    assert "router row published" not in out and "top-k warp" not in out
    assert "ids and weights read" in out
