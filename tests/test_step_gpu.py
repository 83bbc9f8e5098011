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


# ---------------------------------------------------------------- ssd_step_multi: K tokens per call

MULTI = [(64, 1, True, 1), (64, 2, True, 9), (128, 1, True, 16), (128, 4, False, 5), (256, 2, True, 7),
         (512, 1, True, 6), (512, 4, False, 3)]


@pytest.mark.parametrize("N,G,with_D,K", MULTI)
def test_step_multi_equals_repeated_steps(ssd, N, G, with_D, K):
    """K tokens in one call give exactly (bit for bit) what K ssd_step calls give."""
    w, inp = draw(3, K, 8, N, G, seed=21 + N + K, with_D=with_D)
    A = inp["A"].cuda()
    D = None if inp["D"] is None else inp["D"].cuda()
    s_one = inp["init"].clone().cuda()
    ys = []
    for t in range(K):
        x, dt, B, C = token(inp, t)
        ys.append(ssd.ssd_step(x, dt, A, B, C, D, s_one))
    s_multi = inp["init"].clone().cuda()
    y_multi = ssd.ssd_step_multi(inp["x"].cuda(), inp["dt"].cuda(), A, inp["B"].cuda(), inp["C"].cuda(), D, s_multi)
    torch.cuda.synchronize()
    assert torch.equal(y_multi, torch.stack(ys, dim=1))
    assert torch.equal(s_multi, s_one)


@pytest.mark.parametrize("N,G,with_D,K", MULTI)
def test_step_multi_matches_oracle(ssd, N, G, with_D, K):
    w, inp = draw(3, K, 8, N, G, seed=31 + N + K, with_D=with_D)
    ref = oracle_run(w, inp)
    state = inp["init"].clone().cuda()
    D = None if inp["D"] is None else inp["D"].cuda()
    y = ssd.ssd_step_multi(inp["x"].cuda(), inp["dt"].cuda(), inp["A"].cuda(), inp["B"].cuda(), inp["C"].cuda(), D,
                           state)
    torch.cuda.synchronize()
    got = y.float().cpu().numpy().transpose(0, 2, 1, 3).reshape(ref["y"].shape)
    close("y", got, ref["y"])
    close("state", state.cpu().numpy().reshape(ref["final"].shape), ref["final"])


def test_step_multi_continues_forward(ssd):
    """A forward over L tokens, then K more tokens in one multi-token step: the recurrence over L + K."""
    L, K, N = 300, 12, 128
    w, inp = draw(2, L + K, 4, N, 1, seed=13)
    ref = oracle_run(w, inp)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    _, fin = ssd.ssd_forward(d["x"][:, :L].contiguous(), d["dt"][:, :L].contiguous(), d["A"],
                             d["B"][:, :L].contiguous(), d["C"][:, :L].contiguous(), d["D"], d["init"], 128)
    y = ssd.ssd_step_multi(d["x"][:, L:].contiguous(), d["dt"][:, L:].contiguous(), d["A"],
                           d["B"][:, L:].contiguous(), d["C"][:, L:].contiguous(), d["D"], fin)
    torch.cuda.synchronize()
    nunits = w.batch * w.nheads
    got = y.float().cpu().numpy().transpose(0, 2, 1, 3).reshape(nunits, K, 64)
    close("y[L:]", got, ref["y"][:, L:])
    close("state", fin.cpu().numpy().reshape(ref["final"].shape), ref["final"])


def test_step_multi_rejects_bad_arguments(ssd):
    x = torch.zeros((1, 2, 4, 64), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros((1, 4, 64, 64), device="cuda")
    bc = torch.zeros((1, 2, 3, 64), dtype=torch.bfloat16, device="cuda")  # 3 groups do not divide 4 heads
    with pytest.raises(ssd.SSDError):
        ssd.ssd_step_multi(x, torch.zeros((1, 2, 4), device="cuda"), torch.zeros(4, device="cuda"), bc, bc, None, st)


def _misaligned(t):
    """The same values at an address 2 bytes past an 8-byte boundary (the kernels' 2-byte load path)."""
    n = t.numel()
    buf = torch.empty(n + 4, dtype=t.dtype, device=t.device)
    v = buf[1:1 + n].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 8 == 2
    return v


@pytest.mark.parametrize("N", [64, 128, 256])
def test_step_and_multi_bc_alignment_paths_agree(ssd, N):
    """B and C read in 8-byte pieces (aligned) or element by element (2-byte aligned) give the same bits."""
    K = 5
    w, inp = draw(2, K, 4, N, 2, seed=41 + N)
    A, D = inp["A"].cuda(), inp["D"].cuda()
    x, dt = inp["x"].cuda(), inp["dt"].cuda()
    B, C = inp["B"].cuda(), inp["C"].cuda()
    s_a, s_u = inp["init"].clone().cuda(), inp["init"].clone().cuda()
    y_a = ssd.ssd_step_multi(x, dt, A, B, C, D, s_a)
    y_u = ssd.ssd_step_multi(x, dt, A, _misaligned(B), _misaligned(C), D, s_u)
    torch.cuda.synchronize()
    assert torch.equal(y_a, y_u) and torch.equal(s_a, s_u)
    x0, dt0, B0, C0 = token(inp, 0)
    s_a, s_u = inp["init"].clone().cuda(), inp["init"].clone().cuda()
    y_a = ssd.ssd_step(x0, dt0, A, B0, C0, D, s_a)
    y_u = ssd.ssd_step(x0, dt0, A, _misaligned(B0), _misaligned(C0), D, s_u)
    torch.cuda.synchronize()
    assert torch.equal(y_a, y_u) and torch.equal(s_a, s_u)
