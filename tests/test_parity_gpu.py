"""GPU parity: every stage and the whole forward pass against the fp64 oracle.

Tolerance (y, final_state, states): |gpu - ref| <= 1e-2 + 1e-2 * |ref|, element
by element; dA_cumsum: |gpu - ref| <= 1e-5 * |ref| (+1e-30).  Full-size
workloads compare every output of a sample of (batch, head) units, which the
oracle computes one by one (the first and last unit, the first head of every
B/C group, and random ones); small workloads compare everything.
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


def assert_close(name, got, ref, atol=ATOL, rtol=RTOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"got {got[i]} ref {ref[i]} err {err[i]} bound {bound[i]}")


def to_dev(inp):
    return {k: (None if v is None else v.cuda()) for k, v in inp.items()}


def sample_units(w, k, seed=0):
    """k (batch, head) units: the first and the last, the first head of every B/C group (so a
    group-indexing slip in any group shows), and random ones for the rest."""
    n = w.batch * w.nheads
    if k >= n:
        return np.arange(n)
    rng = np.random.default_rng(seed)
    hpg = w.nheads // w.ngroups
    u = set([0, n - 1]) | {g * hpg for g in range(w.ngroups)}
    while len(u) < k:
        u.add(int(rng.integers(0, n)))
    return np.array(sorted(u))


def unit_rows(t, w, units):
    """(batch, L, H, P) tensor -> (nunits, L, P) rows of the sampled units."""
    t = t.float().cpu().numpy() if torch.is_tensor(t) else t
    return np.stack([t[u // w.nheads, :, u % w.nheads] for u in units])


def unit_states(t, w, units):
    """(batch, H, P, N) tensor -> (nunits, P, N)."""
    t = t.cpu().numpy()
    return np.stack([t[u // w.nheads, u % w.nheads] for u in units])


def unit_chunk_states(t, w, units):
    """(batch, nc, H, P, N) tensor -> (nunits, nc, P, N)."""
    t = t.cpu().numpy()
    return np.stack([t[u // w.nheads, :, u % w.nheads] for u in units])


# name -> number of sampled units (None = all)
FULL = [("tiny_L512_N64", None), ("mamba2_1p3b_layer_2x4096_N128", 24), ("long_L65536_N128", 4),
        ("state_sweep_L16384_N64", 6), ("state_sweep_L16384_N128", 6), ("state_sweep_L16384_N256", 6),
        ("state_sweep_L16384_N512", 4), ("longest_L262144_N256_G8", 3)]


@pytest.mark.parametrize("name,k", FULL)
def test_forward_workloads(ssd, name, k):
    w = I.WORKLOADS[name]
    inp = I.make_inputs(w, seed=0)
    d = to_dev(inp)
    y, fin = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], w.chunk_size)
    torch.cuda.synchronize()
    assert ssd.ssd_get_device_error() == 0
    units = sample_units(w, k if k is not None else w.batch * w.nheads)
    n = I.as_numpy(inp)
    ref = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], w.chunk_size, units=units)
    assert_close(f"{name} y", unit_rows(y, w, units), ref["y"])
    assert_close(f"{name} final", unit_states(fin, w, units), ref["final"])


EDGE = [
    # (batch, L, H, N, G, Q, init, with_D)
    (1, 1, 2, 64, 1, 64, True, True),        # a single token
    (1, 63, 2, 64, 2, 64, False, True),      # L < Q, G = H
    (2, 300, 4, 128, 2, 256, True, True),    # ragged tail, two groups
    (1, 1000, 3, 256, 1, 128, True, False),  # odd H, no D, ragged
    (1, 513, 2, 512, 1, 256, True, True),    # largest state, ragged
    (3, 257, 8, 64, 4, 64, False, True),     # batch 3, several groups, ragged by one
]


@pytest.mark.parametrize("b,L,H,N,G,Q,init,with_D", EDGE)
def test_forward_edge_cases(ssd, b, L, H, N, G, Q, init, with_D):
    w = I.Workload("edge", b, L, H, 64, N, G, Q, init)
    inp = I.make_inputs(w, seed=3)
    if not with_D:
        inp["D"] = None
    d = to_dev(inp)
    y, fin = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], Q)
    torch.cuda.synchronize()
    n = I.as_numpy(inp)
    ref = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], Q)
    units = np.arange(b * H)
    assert_close("y", unit_rows(y, w, units), ref["y"])
    assert_close("final", unit_states(fin, w, units), ref["final"])


LONG_RAGGED = [
    # (batch, L, H, N, G, Q): enough (batch, head, chunk) units that ssd_forward runs compute_out over
    # spans of several span-start states, with a ragged tail (L % Q != 0) and a short last span
    (1, 65536 - 100, 32, 64, 1, 256),
    (2, 16384 + 64 + 7, 16, 128, 2, 128),
    (1, 32768 - 1, 24, 256, 3, 64),
]


@pytest.mark.parametrize("b,L,H,N,G,Q", LONG_RAGGED)
def test_forward_long_ragged(ssd, b, L, H, N, G, Q):
    w = I.Workload("long_ragged", b, L, H, 64, N, G, Q, True)
    inp = I.make_inputs(w, seed=5)
    d = to_dev(inp)
    y, fin = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], Q)
    torch.cuda.synchronize()
    assert ssd.ssd_get_device_error() == 0
    units = sample_units(w, 5, seed=b + H)
    n = I.as_numpy(inp)
    ref = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], Q, units=units)
    assert_close("y", unit_rows(y, w, units), ref["y"])
    assert_close("final", unit_states(fin, w, units), ref["final"])


@pytest.mark.parametrize("Q", [64, 128, 256])
def test_chunk_size_invariance(ssd, Q):
    """The same sequence at every chunk size gives the recurrence's y (P4 on the GPU)."""
    w = I.Workload("inv", 1, 1100, 4, 64, 128, 1, Q, True)
    inp = I.make_inputs(w, seed=5)
    d = to_dev(inp)
    y, fin = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], Q)
    n = I.as_numpy(inp)
    ref = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], 64)
    units = np.arange(4)
    assert_close("y", unit_rows(y, w, units), ref["y"])
    assert_close("final", unit_states(fin, w, units), ref["final"])


def test_large_decay_memoryless(ssd):
    """Huge |A| dt: every token forgets its past; exp2 arguments reach far below -126."""
    w = I.Workload("decay", 1, 700, 4, 64, 128, 1, 256, True)
    inp = I.make_inputs(w, seed=7)
    inp["A"] = torch.full_like(inp["A"], -1.0e3)
    d = to_dev(inp)
    y, fin = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], 256)
    n = I.as_numpy(inp)
    ref = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], 256)
    units = np.arange(4)
    assert_close("y", unit_rows(y, w, units), ref["y"])
    assert_close("final", unit_states(fin, w, units), ref["final"])


def test_no_final_state(ssd):
    w = I.WORKLOADS["tiny_L512_N64"]
    inp = I.make_inputs(w, seed=0)
    d = to_dev(inp)
    y, fin = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], w.chunk_size,
                             want_final=False)
    assert fin is None
    n = I.as_numpy(inp)
    ref = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], w.chunk_size)
    assert_close("y", unit_rows(y, w, np.arange(4)), ref["y"])


# --------------------------------------------------------------- stages

STAGE = [("tiny_L512_N64", None), ("mamba2_1p3b_layer_2x4096_N128", 8), ("state_sweep_L16384_N512", 3),
         ("long_L65536_N128", 3)]


@pytest.mark.parametrize("name,k", STAGE + [("longest_L262144_N256_G8", 2)])
def test_stage_chunk_cumsum(ssd, name, k):
    w = I.WORKLOADS[name]
    inp = I.make_inputs(w, seed=0)
    cs, dtt = ssd.ssd_chunk_cumsum(inp["dt"].cuda(), inp["A"].cuda(), w.chunk_size)
    rcs, rdt = oracle.dA_cumsum(inp["dt"].numpy(), inp["A"].numpy(), w.chunk_size)
    assert_close("dA_cumsum", cs.cpu().numpy(), rcs, atol=1e-30, rtol=1e-5)
    np.testing.assert_array_equal(dtt.cpu().numpy(), rdt.astype(np.float32))


def test_stage_chunk_cumsum_ragged(ssd):
    for L, Q in ((1, 64), (100, 64), (333, 128), (257, 256)):
        g = torch.Generator().manual_seed(L)
        dt = torch.nn.functional.softplus(torch.randn((2, L, 37), generator=g) - 4)
        A = -torch.exp(torch.rand(37, generator=g) * 2.77)
        cs, dtt = ssd.ssd_chunk_cumsum(dt.cuda(), A.cuda(), Q)
        rcs, rdt = oracle.dA_cumsum(dt.numpy(), A.numpy(), Q)
        assert_close(f"cs L={L}", cs.cpu().numpy(), rcs, atol=1e-30, rtol=1e-5)
        np.testing.assert_array_equal(dtt.cpu().numpy(), rdt.astype(np.float32))


@pytest.mark.parametrize("name,k", STAGE)
def test_stage_chunk_state(ssd, name, k):
    w = I.WORKLOADS[name]
    inp = I.make_inputs(w, seed=0)
    n = I.as_numpy(inp)
    rcs, rdt = oracle.dA_cumsum(n["dt"], n["A"], w.chunk_size)
    cs = torch.from_numpy(rcs.astype(np.float32)).cuda()
    dtt = torch.from_numpy(rdt.astype(np.float32)).cuda()
    S = ssd.ssd_chunk_state(inp["x"].cuda(), inp["B"].cuda(), dtt, cs, w.chunk_size)
    units = sample_units(w, k if k is not None else w.batch * w.nheads)
    ref = oracle.chunk_states(n["x"], n["dt"], n["A"], n["B"], w.chunk_size, units=units)
    assert_close("chunk_states", unit_chunk_states(S, w, units), ref)


@pytest.mark.parametrize("name,k", STAGE)
def test_stage_state_passing(ssd, name, k):
    w = I.WORKLOADS[name]
    g = torch.Generator().manual_seed(11)
    nc = w.nchunks
    S = torch.randn((w.batch, nc, w.nheads, w.headdim, w.dstate), generator=g)
    cs = -torch.rand((w.batch, w.nheads, nc, w.chunk_size), generator=g) * 4
    init = torch.randn((w.batch, w.nheads, w.headdim, w.dstate), generator=g)
    states, fin = ssd.ssd_state_passing(S.cuda(), cs.cuda(), init.cuda(), w.chunk_size)
    rst, rfin = oracle.state_passing(S.numpy(), cs.numpy(), init.numpy(), w.chunk_size)
    assert_close("states", states.cpu().numpy(), rst, atol=1e-5, rtol=1e-5)
    assert_close("final", fin.cpu().numpy(), rfin, atol=1e-5, rtol=1e-5)
    # in place (states aliasing chunk_states), no init, no final
    Sd = S.cuda()
    ssd.ssd_state_passing(Sd, cs.cuda(), None, w.chunk_size, states=Sd, want_final=False)
    rst0, _ = oracle.state_passing(S.numpy(), cs.numpy(), None, w.chunk_size)
    assert_close("states in place", Sd.cpu().numpy(), rst0, atol=1e-5, rtol=1e-5)


@pytest.mark.parametrize("name,k", STAGE)
def test_stage_chunk_scan(ssd, name, k):
    w = I.WORKLOADS[name]
    inp = I.make_inputs(w, seed=0)
    n = I.as_numpy(inp)
    units = sample_units(w, k if k is not None else w.batch * w.nheads)
    # chunk-start states: oracle states for the sampled units, random elsewhere
    g = torch.Generator().manual_seed(3)
    states = 0.3 * torch.randn((w.batch, w.nchunks, w.nheads, w.headdim, w.dstate), generator=g)
    o = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], w.chunk_size, units=units,
                       want_chunk_starts=True)
    for i, u in enumerate(units):
        states[u // w.nheads, :, u % w.nheads] = torch.from_numpy(o["chunk_starts"][i].astype(np.float32))
    rcs, rdt = oracle.dA_cumsum(n["dt"], n["A"], w.chunk_size)
    y = ssd.ssd_chunk_scan(inp["x"].cuda(), inp["B"].cuda(), inp["C"].cuda(),
                           torch.from_numpy(rdt.astype(np.float32)).cuda(),
                           torch.from_numpy(rcs.astype(np.float32)).cuda(), inp["D"].cuda(), states.cuda(),
                           w.chunk_size)
    ref = oracle.chunk_scan(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], states.numpy(), w.chunk_size,
                            units=units)
    assert_close("y", unit_rows(y, w, units), ref)


def test_pipeline_of_stages_matches_forward(ssd):
    """The four stage entry points chained by hand give the oracle's y."""
    w = I.WORKLOADS["mamba2_1p3b_layer_2x4096_N128"]
    inp = I.make_inputs(w, seed=1)
    d = to_dev(inp)
    cs, dtt = ssd.ssd_chunk_cumsum(d["dt"], d["A"], w.chunk_size)
    S = ssd.ssd_chunk_state(d["x"], d["B"], dtt, cs, w.chunk_size)
    st, fin = ssd.ssd_state_passing(S, cs, d["init"], w.chunk_size)
    y = ssd.ssd_chunk_scan(d["x"], d["B"], d["C"], dtt, cs, d["D"], st, w.chunk_size)
    units = sample_units(w, 8)
    n = I.as_numpy(inp)
    ref = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], w.chunk_size, units=units)
    assert_close("y", unit_rows(y, w, units), ref["y"])
    assert_close("final", unit_states(fin, w, units), ref["final"])


def test_nonblocking_stream(ssd):
    """Work issued on a side stream is ordered on that stream."""
    w = I.WORKLOADS["tiny_L512_N64"]
    inp = I.make_inputs(w, seed=2)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = to_dev(inp)
        y, fin = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], w.chunk_size, stream=s)
    s.synchronize()
    n = I.as_numpy(inp)
    ref = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], w.chunk_size)
    assert_close("y", unit_rows(y, w, np.arange(4)), ref["y"])


@pytest.mark.parametrize("name", ["mamba2_1p3b_layer_2x4096_N128", "state_sweep_L16384_N512"])
def test_forward_y_alignment_paths_agree(ssd, name):
    """y rows stored in 32-byte pieces (y 32-byte aligned) or 16-byte pieces (y only 16-byte aligned):
    the same bits either way."""
    w = I.WORKLOADS[name]
    d = to_dev(I.make_inputs(w, seed=2))
    y_a, _ = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], w.chunk_size)
    buf = torch.empty(d["x"].numel() + 16, dtype=torch.bfloat16, device="cuda")
    y_u = buf[8:8 + d["x"].numel()].view(d["x"].shape)
    assert y_u.data_ptr() % 32 == 16
    ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], w.chunk_size, y=y_u)
    torch.cuda.synchronize()
    assert ssd.ssd_get_device_error() == 0
    assert torch.equal(y_a, y_u)
