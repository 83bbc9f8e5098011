"""The failure path of the pipelined tensor-core kernels, made to run on purpose
without faulting or hanging the GPU.

ssd_debug_stall makes the selected kernels first wait on a barrier that
nothing completes; with a 2 ms wait limit that wait runs out, the kernel sets
its error word, every role abandons its work, the teardown drains let the
copies and products already issued finish, and the kernel returns.  The test
then checks that the host sees SSD_ERR_TIMEOUT, that the device is still
usable, and that the next normal call matches the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from state_space_sequence_ssd_gb300 import _ffi
from state_space_sequence_ssd_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssd():
    from state_space_sequence_ssd_gb300 import build
    build.build()
    import state_space_sequence_ssd_gb300 as m
    m.ssd_get_device_error()
    yield m
    lib = _ffi.lib()
    lib.ssd_debug_stall(0)
    lib.ssd_debug_set_wait_limit_ns(0)


def kind(lib, name):
    for k in range(16):
        if lib.ssd_kernel_name(k).decode() == name:
            return k
    raise KeyError(name)


def forward(ssd, w, d):
    return ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], w.chunk_size)


@pytest.mark.parametrize("stage", ["chunk_state", "chunk_scan"])
@pytest.mark.parametrize("name", ["tiny_L512_N64", "mamba2_1p3b_layer_2x4096_N128"])
def test_stalled_wait_times_out_and_the_device_recovers(ssd, stage, name):
    lib = _ffi.lib()
    w = I.WORKLOADS[name]
    inp = I.make_inputs(w, seed=41)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    assert lib.ssd_debug_set_wait_limit_ns(2_000_000) == 0
    assert lib.ssd_debug_stall(1 << kind(lib, stage)) == 0
    try:
        forward(ssd, w, d)  # launches succeed; the stalled kernel gives up on the device
        torch.cuda.synchronize()
        assert ssd.ssd_get_device_error() == _ffi.SSD_ERR_TIMEOUT
    finally:
        lib.ssd_debug_stall(0)
        lib.ssd_debug_set_wait_limit_ns(0)
    assert ssd.ssd_get_device_error() == 0, "reading the error words clears them"
    y, fin = forward(ssd, w, d)
    torch.cuda.synchronize()
    assert ssd.ssd_get_device_error() == 0
    units = np.array([0, w.batch * w.nheads - 1])
    n = I.as_numpy(inp)
    ref = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], w.chunk_size, units=units)
    got_y = np.stack([y[u // w.nheads, :, u % w.nheads].float().cpu().numpy() for u in units])
    got_f = np.stack([fin[u // w.nheads, u % w.nheads].cpu().numpy() for u in units])
    for name_, got, want in (("y", got_y, ref["y"]), ("final", got_f, ref["final"])):
        err = np.abs(got - want)
        assert (err <= 1e-2 + 1e-2 * np.abs(want)).all(), f"{name_}: max err {err.max()}"


def test_short_limit_alone_does_not_break_a_normal_call(ssd):
    """A 50 ms limit is far above any wait of a healthy pipeline: no report, right result."""
    lib = _ffi.lib()
    w = I.WORKLOADS["tiny_L512_N64"]
    inp = I.make_inputs(w, seed=42)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    lib.ssd_debug_set_wait_limit_ns(50_000_000)
    try:
        y, _ = forward(ssd, w, d)
        torch.cuda.synchronize()
        assert ssd.ssd_get_device_error() == 0
    finally:
        lib.ssd_debug_set_wait_limit_ns(0)
    n = I.as_numpy(inp)
    ref = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], w.chunk_size)
    got = np.stack([y[0, :, h].float().cpu().numpy() for h in range(w.nheads)])
    assert (np.abs(got - ref["y"]) <= 1e-2 + 1e-2 * np.abs(ref["y"])).all()


@pytest.mark.parametrize("name", ["tiny_L512_N64", "mamba2_1p3b_layer_2x4096_N128"])
def test_backward_stall_times_out_and_the_device_recovers(ssd, name):
    """The backward kernel (clusters of CTAs over a group's heads at these shapes) gives up on a stalled
    wait: every CTA still meets the cluster barriers, the host sees SSD_ERR_TIMEOUT, and the next call is
    right."""
    lib = _ffi.lib()
    w = I.WORKLOADS[name]
    inp = I.make_inputs(w, seed=43)
    gr = I.make_grad_inputs(w, seed=43)
    d = {k: (None if v is None else v.cuda()) for k, v in {**inp, **gr}.items()}

    def backward():
        return ssd.ssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], d["dy"], d["dfinal"],
                                chunk_size=w.chunk_size)

    assert lib.ssd_debug_set_wait_limit_ns(2_000_000) == 0
    assert lib.ssd_debug_stall(1 << kind(lib, "bwd_chunk")) == 0
    try:
        backward()
        torch.cuda.synchronize()
        assert ssd.ssd_get_device_error() == _ffi.SSD_ERR_TIMEOUT
    finally:
        lib.ssd_debug_stall(0)
        lib.ssd_debug_set_wait_limit_ns(0)
    assert ssd.ssd_get_device_error() == 0
    out = backward()
    torch.cuda.synchronize()
    assert ssd.ssd_get_device_error() == 0
    units = np.array([0, w.batch * w.nheads - 1])
    n = I.as_numpy(inp)
    g = I.as_numpy(gr)
    r = oracle.backward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], g["dy"], g["dfinal"],
                        units=units, scales=True)
    got = np.stack([out["dx"][u // w.nheads, :, u % w.nheads].float().cpu().numpy() for u in units])
    err = np.abs(got - r["dx"])
    assert (err <= 1e-2 + 1e-2 * np.abs(r["dx"]) + 2.0 ** -9 * r["dx_s"]).all(), f"dx: max err {err.max()}"
