"""The head-partitioned split on one GPU: ssd_forward_heads over the parts that ssd_partition_heads gives
for 2, 3 and 4 devices, run one after the other into the same full-size outputs, equals the whole
problem -- against the oracle at the path's tolerance, and against one whole-problem ssd_forward.  A
part writes only its own heads' rows of y and final_state."""
import numpy as np
import pytest
import torch

import oracle
from state_space_sequence_ssd_gb300 import inputs as I

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 1e-2


@pytest.fixture(scope="module")
def ssd():
    from state_space_sequence_ssd_gb300 import build
    build.build()
    import state_space_sequence_ssd_gb300 as m
    m.ssd_get_device_error()
    return m


def close(name, got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{name}: {bad.sum()} of {bad.size} outside tolerance, max err {err.max()}"


CASES = [
    # (batch, L, H, N, G, Q, nparts)
    (2, 1024, 16, 128, 1, 256, 2),   # one group split across two devices (two-head compute_out)
    (1, 2000, 12, 128, 1, 128, 3),   # three parts, ragged tail
    (1, 1536, 16, 64, 4, 64, 4),     # whole groups per device
    (1, 777, 6, 256, 3, 128, 2),     # dstate 256 (one head per CTA), groups split 1 / 2
    (1, 640, 10, 64, 5, 64, 3),      # odd heads per group (one head per CTA)
]


@pytest.mark.parametrize("b,L,H,N,G,Q,nparts", CASES)
def test_parts_compose_the_whole_forward(ssd, b, L, H, N, G, Q, nparts):
    w = I.Workload("heads", b, L, H, 64, N, G, Q, True)
    inp = I.make_inputs(w, seed=51)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    y = torch.full_like(d["x"], float("nan"))
    fin = torch.full((b, H, 64, N), float("nan"), device="cuda")
    parts = [ssd.ssd_partition_heads(H, G, nparts, p) for p in range(nparts)]
    for k, (hb, hc) in enumerate(parts):
        if hc == 0:
            continue
        ssd.ssd_forward_heads(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], Q, hb, hc, y=y,
                              final_state=fin)
        torch.cuda.synchronize()
        assert ssd.ssd_get_device_error() == 0
        done = sum(c for _, c in parts[:k + 1])
        # the heads of later parts are still untouched
        assert bool(torch.isnan(y[:, :, done:].float()).all()) and bool(torch.isnan(fin[:, done:]).all())
    y_ref, fin_ref = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], Q)
    torch.cuda.synchronize()
    close("y vs ssd_forward", y.float().cpu().numpy(), y_ref.float().cpu().numpy())
    close("final vs ssd_forward", fin.cpu().numpy(), fin_ref.cpu().numpy())
    n = I.as_numpy(inp)
    units = np.arange(b * H)
    ref = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], Q, units=units)
    got_y = np.stack([y[u // H, :, u % H].float().cpu().numpy() for u in units])
    got_f = np.stack([fin[u // H, u % H].cpu().numpy() for u in units])
    close("y vs oracle", got_y, ref["y"])
    close("final vs oracle", got_f, ref["final"])


def test_whole_range_is_ssd_forward(ssd):
    """head_begin 0, head_count nheads: the same call as ssd_forward, bit for bit."""
    w = I.WORKLOADS["mamba2_1p3b_layer_2x4096_N128"]
    d = {k: (None if v is None else v.cuda()) for k, v in I.make_inputs(w, seed=52).items()}
    y1, f1 = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], w.chunk_size)
    y2, f2 = ssd.ssd_forward_heads(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], w.chunk_size,
                                   0, w.nheads)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(f1, f2)
