"""GPU parity of ssd_step (one recurrent step) against the fp64 oracle.

The oracle's recurrence over one token with a given initial state is the
step's definition; chaining steps must reproduce the recurrence over many
tokens, and a step after ssd_forward must continue the forward pass exactly
(the state hand-off of the recurrent mode).  Tolerance as for the forward
pass: |gpu - ref| <= 1e-2 + 1e-2 |ref|.
"""
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
    return m


def close(name, got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), name
    bad = np.abs(got - ref) > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{name}: {bad.sum()} of {bad.size} outside tolerance, max err {np.abs(got - ref).max()}"


def draw(batch, L, H, N, G, seed, with_D=True):
    w = I.Workload("step", batch, L, H, 64, N, G, 64, True)
    inp = I.make_inputs(w, seed=seed)
    if not with_D:
        inp["D"] = None
    return w, inp


def oracle_run(w, inp):
    n = I.as_numpy(inp)
    return oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], w.chunk_size)


def token(inp, t):
    """Inputs of token t as the step's (batch, ...) tensors on the GPU."""
    return (inp["x"][:, t].contiguous().cuda(), inp["dt"][:, t].contiguous().cuda(), inp["B"][:, t].contiguous().cuda(),
            inp["C"][:, t].contiguous().cuda())


@pytest.mark.parametrize("N,G,with_D", [(64, 1, True), (128, 2, True), (256, 1, False), (512, 4, True)])
def test_step_matches_oracle(ssd, N, G, with_D):
    w, inp = draw(3, 1, 8, N, G, seed=11 + N, with_D=with_D)
    ref = oracle_run(w, inp)
    x, dt, B, C = token(inp, 0)
    state = inp["init"].clone().cuda()
    D = None if inp["D"] is None else inp["D"].cuda()
    y = ssd.ssd_step(x, dt, inp["A"].cuda(), B, C, D, state)
    torch.cuda.synchronize()
    close("y", y.float().cpu().numpy().reshape(ref["y"].shape), ref["y"])
    close("state", state.cpu().numpy().reshape(ref["final"].shape), ref["final"])


@pytest.mark.parametrize("N", [64, 128])
def test_chained_steps_equal_the_recurrence(ssd, N):
    L = 16
    w, inp = draw(2, L, 4, N, 1, seed=5)
    ref = oracle_run(w, inp)
    state = inp["init"].clone().cuda()
    A = inp["A"].cuda()
    D = inp["D"].cuda()
    ys = []
    for t in range(L):
        x, dt, B, C = token(inp, t)
        ys.append(ssd.ssd_step(x, dt, A, B, C, D, state).float().cpu())
    torch.cuda.synchronize()
    y = torch.stack(ys, dim=1).numpy()  # (b, L, H, P)
    got = y.transpose(0, 2, 1, 3).reshape(ref["y"].shape)
    close("y", got, ref["y"])
    close("state", state.cpu().numpy().reshape(ref["final"].shape), ref["final"])


@pytest.mark.parametrize("N,Q", [(64, 64), (128, 128)])
def test_step_continues_forward(ssd, N, Q):
    L = 300  # ragged: not a multiple of the chunk size
    w, inp = draw(2, L + 1, 4, N, 1, seed=9)
    ref = oracle_run(w, inp)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    y_fw, fin = ssd.ssd_forward(d["x"][:, :L].contiguous(), d["dt"][:, :L].contiguous(), d["A"],
                                d["B"][:, :L].contiguous(), d["C"][:, :L].contiguous(), d["D"], d["init"], Q)
    x, dt, B, C = token(inp, L)
    y_st = ssd.ssd_step(x, dt, d["A"], B, C, d["D"], fin)
    torch.cuda.synchronize()
    nunits = w.batch * w.nheads
    ref_last = ref["y"][:, L]  # (nunits, P)
    close("y[L]", y_st.float().cpu().numpy().reshape(nunits, 64), ref_last)
    close("state", fin.cpu().numpy().reshape(ref["final"].shape), ref["final"])


def test_step_rejects_bad_arguments(ssd):
    x = torch.zeros((1, 4, 64), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros((1, 4, 64, 64), device="cuda")
    with pytest.raises(ssd.SSDError):
        ssd.ssd_step(x, torch.zeros((1, 4), device="cuda"), torch.zeros(4, device="cuda"),
                     torch.zeros((1, 3, 64), dtype=torch.bfloat16, device="cuda"),  # 3 groups do not divide 4 heads
                     torch.zeros((1, 3, 64), dtype=torch.bfloat16, device="cuda"), None, st)
