"""GPU parity of the input-side options (ssd_forward_ex, ssd_step_ex) against the fp64 oracle.

dt <- clamp(softplus(dt + dt_bias)), one skip weight per channel (D is (H, P)) and the output gate
y <- y z sigmoid(z), each alone and all together, at sizes that span several 128-token sub-blocks,
several chunks per span and a ragged tail.  Tolerance as for the forward pass:
|gpu - ref| <= 1e-2 + 1e-2 |ref|.
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
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{name}: {bad.sum()} of {bad.size} outside tolerance, max err {err.max()}"


def rows(y, w, units=None):
    """(batch, L, H, P) -> (units, L, P) as the oracle orders them."""
    y = y.float().cpu().numpy().transpose(0, 2, 1, 3).reshape(w.batch * w.nheads, w.seqlen, w.headdim)
    return y if units is None else y[units]


OPTION_SETS = {
    "bias_softplus": dict(dt_bias=True, dt_softplus=True),
    "limit": dict(dt_bias=True, dt_softplus=True, dt_limit=True),
    "D_per_channel": dict(D_hp=True),
    "z_gate": dict(z=True),
    "all": dict(dt_bias=True, dt_softplus=True, dt_limit=True, D_hp=True, z=True),
}


def case(w, which, seed=0):
    inp = I.make_inputs(w, seed=seed)
    lo = I.make_layer_options(w, seed=seed)
    sel = OPTION_SETS[which]
    dt = lo["dt_raw"] if sel.get("dt_softplus") else inp["dt"]
    kw = dict(dt_bias=lo["dt_bias"] if sel.get("dt_bias") else None, dt_softplus=bool(sel.get("dt_softplus")),
              dt_limit=lo["dt_limit"] if sel.get("dt_limit") else None, z=lo["z"] if sel.get("z") else None)
    D = lo["D_hp"] if sel.get("D_hp") else inp["D"]
    return inp, dt, D, kw


def oracle_run(w, inp, dt, D, kw, units=None):
    n = I.as_numpy(inp)
    okw = dict(kw)
    okw["dt_bias"] = None if kw["dt_bias"] is None else kw["dt_bias"].numpy()
    okw["z"] = None if kw["z"] is None else I.bf16_bits(kw["z"])
    return oracle.forward(n["x"], dt.numpy(), n["A"], n["B"], n["C"], D.numpy(), n["init"], w.chunk_size,
                          units=units, **okw)


def gpu_run(ssd, w, inp, dt, D, kw):
    dv = lambda t: None if t is None else t.cuda()
    return ssd.ssd_forward_ex(dv(inp["x"]), dv(dt), dv(inp["A"]), dv(inp["B"]), dv(inp["C"]), dv(D), dv(inp["init"]),
                              w.chunk_size, dt_bias=dv(kw["dt_bias"]), dt_softplus=kw["dt_softplus"],
                              dt_limit=kw["dt_limit"], z=dv(kw["z"]))


@pytest.mark.parametrize("which", sorted(OPTION_SETS))
@pytest.mark.parametrize("N,Q,G", [(64, 64, 2), (128, 256, 1)])
def test_forward_ex_matches_oracle(ssd, which, N, Q, G):
    w = I.Workload("opts", 2, 1000, 4, 64, N, G, Q, True)  # ragged: 1000 = 3 x 256 + 232
    inp, dt, D, kw = case(w, which, seed=N)
    ref = oracle_run(w, inp, dt, D, kw)
    y, fin = gpu_run(ssd, w, inp, dt, D, kw)
    torch.cuda.synchronize()
    close("y", rows(y, w), ref["y"])
    close("final", fin.cpu().numpy().reshape(ref["final"].shape), ref["final"])


@pytest.mark.parametrize("N", [256, 512])
def test_forward_ex_all_options_large_state(ssd, N):
    w = I.Workload("opts", 1, 600, 4, 64, N, 1, 256, True)
    inp, dt, D, kw = case(w, "all", seed=3)
    ref = oracle_run(w, inp, dt, D, kw)
    y, fin = gpu_run(ssd, w, inp, dt, D, kw)
    torch.cuda.synchronize()
    close("y", rows(y, w), ref["y"])
    close("final", fin.cpu().numpy().reshape(ref["final"].shape), ref["final"])


def test_forward_ex_without_options_is_forward(ssd):
    w = I.WORKLOADS["tiny_L512_N64"]
    inp = {k: (None if v is None else v.cuda()) for k, v in I.make_inputs(w, seed=4).items()}
    a = ssd.ssd_forward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["init"], w.chunk_size)
    b = ssd.ssd_forward_ex(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["init"], w.chunk_size)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_forward_ex_all_options_mamba2_layer_sampled(ssd):
    """The 1.3B-layer workload (2 x 4096 tokens, 64 heads, N 128) with every option, sampled (batch, head) units."""
    w = I.WORKLOADS["mamba2_1p3b_layer_2x4096_N128"]
    inp, dt, D, kw = case(w, "all", seed=5)
    units = np.array([0, 17, 63, 64, 100, 127])
    ref = oracle_run(w, inp, dt, D, kw, units=units)
    y, fin = gpu_run(ssd, w, inp, dt, D, kw)
    torch.cuda.synchronize()
    close("y", rows(y, w, units), ref["y"])
    finn = fin.cpu().numpy().reshape(w.batch * w.nheads, w.headdim, w.dstate)[units]
    close("final", finn, ref["final"])


@pytest.mark.parametrize("which", sorted(OPTION_SETS))
@pytest.mark.parametrize("N", [64, 256])
def test_step_ex_matches_oracle(ssd, which, N):
    w = I.Workload("opts_step", 3, 1, 8, 64, N, 2, 64, True)
    inp, dt, D, kw = case(w, which, seed=20 + N)
    ref = oracle_run(w, inp, dt, D, kw)
    state = inp["init"].clone().cuda()
    dv = lambda t: None if t is None else t.cuda()
    y = ssd.ssd_step_ex(inp["x"][:, 0].contiguous().cuda(), dt[:, 0].contiguous().cuda(), dv(inp["A"]),
                        inp["B"][:, 0].contiguous().cuda(), inp["C"][:, 0].contiguous().cuda(), dv(D), state,
                        dt_bias=dv(kw["dt_bias"]), dt_softplus=kw["dt_softplus"], dt_limit=kw["dt_limit"],
                        z=None if kw["z"] is None else kw["z"][:, 0].contiguous().cuda())
    torch.cuda.synchronize()
    close("y", y.float().cpu().numpy().reshape(ref["y"].shape), ref["y"])
    close("state", state.cpu().numpy().reshape(ref["final"].shape), ref["final"])


def test_step_ex_continues_forward_ex(ssd):
    """A layer with every option: ssd_forward_ex over L tokens, then ssd_step_ex on token L, equals L + 1 tokens."""
    L = 200
    w = I.Workload("opts_chain", 2, L + 1, 4, 64, 128, 1, 64, True)
    inp, dt, D, kw = case(w, "all", seed=8)
    ref = oracle_run(w, inp, dt, D, kw)
    c = lambda t: t.contiguous().cuda()
    y_fw, fin = ssd.ssd_forward_ex(c(inp["x"][:, :L]), c(dt[:, :L]), c(inp["A"]), c(inp["B"][:, :L]),
                                   c(inp["C"][:, :L]), c(D), c(inp["init"]), 64, dt_bias=c(kw["dt_bias"]),
                                   dt_softplus=True, dt_limit=kw["dt_limit"], z=c(kw["z"][:, :L]))
    y_st = ssd.ssd_step_ex(c(inp["x"][:, L]), c(dt[:, L]), c(inp["A"]), c(inp["B"][:, L]), c(inp["C"][:, L]), c(D),
                           fin, dt_bias=c(kw["dt_bias"]), dt_softplus=True, dt_limit=kw["dt_limit"],
                           z=c(kw["z"][:, L]))
    torch.cuda.synchronize()
    close("y[:L]", rows(y_fw, w.with_(seqlen=L)), ref["y"][:, :L])
    close("y[L]", y_st.float().cpu().numpy().reshape(w.batch * w.nheads, 64), ref["y"][:, L])
    close("state", fin.cpu().numpy().reshape(ref["final"].shape), ref["final"])


def _offset16(t):
    """The same values at an address 16 bytes past a 32-byte boundary."""
    n = t.numel()
    buf = torch.empty(n + 16, dtype=t.dtype, device=t.device)
    v = buf[8:8 + n].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 32 == 16
    return v


def test_forward_ex_gate_and_y_alignment_paths_agree(ssd):
    """z rows loaded and y rows stored in 32-byte pieces (32-byte aligned) or 16-byte pieces (16-byte
    aligned only): the same bits."""
    w = I.WORKLOADS["mamba2_1p3b_layer_2x4096_N128"]
    inp, dt, D, kw = case(w, "all", seed=6)
    dv = lambda t: None if t is None else t.cuda()
    args = (dv(inp["x"]), dv(dt), dv(inp["A"]), dv(inp["B"]), dv(inp["C"]), dv(D), dv(inp["init"]), w.chunk_size)
    z = dv(kw["z"])
    opt = dict(dt_bias=dv(kw["dt_bias"]), dt_softplus=kw["dt_softplus"], dt_limit=kw["dt_limit"])
    y_a, f_a = ssd.ssd_forward_ex(*args, z=z, **opt)
    y_u = _offset16(torch.zeros_like(y_a))
    _, f_u = ssd.ssd_forward_ex(*args, z=_offset16(z), y=y_u, **opt)
    torch.cuda.synchronize()
    assert ssd.ssd_get_device_error() == 0
    assert torch.equal(y_a, y_u) and torch.equal(f_a, f_u)
