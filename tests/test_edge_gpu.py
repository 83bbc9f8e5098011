"""GPU parity on the method's own edge cases and at the edge of float16's range.

* A = 0: no decay, so the state after a run of tokens is the pages' jump
  formula h(t+T) = h(t) + B X^T with X's rows scaled by dt
  (disconfirmai.com page "Jane Street ML Engineers Map Mamba-2 Recurrent
  State Computation to Tensor Cores with cuTile", jump-formula paragraph).
  final_state is checked against that formula written out in numpy, and y
  and final_state against the oracle.
* dt = 0 on a whole chunk and on the last token of a ragged tail (the
  zero-padding reading of the devotd.net page's chunk_cumsum listing), and
  dt = 0 everywhere, where y = C . init + D x and final_state = init exactly.
* Magnitude sweep: x, B and C scaled by 8, 64 and 256 with |A| of 1e-3 and
  1.  The tensor-core operands are float16, so large enough inputs push a
  converted value (an input, an entry of the masked matrix, of the carried
  state or of a scaled x row) past 65504.  Every call must then either match
  the oracle or report SSD_ERR_RANGE -- never a silently wrong result.

Tolerance.  The elementwise bound |gpu - ref| <= 1e-2 + 1e-2 |ref| holds on the
five workloads and on every case whose outputs have an RMS of order one.  The
decay-free sum over 16384 tokens and the scaled inputs push the output's RMS
to 50-10^4, where float16 rounding of the tensor-core operands (relative error
<= 2^-11 on the carried state, on the scaled x rows and on the masked matrix)
gives errors proportional to the size of the terms, not of the result: where
y is a cancellation of large terms the fixed 1e-2 floor is below that
rounding.  Those cases are checked against the derived bound
    |gpu - ref| <= 1e-2 + 1e-2 |ref| + 3e-3 * rms(ref of the (batch, head) unit):
three roundings of 2^-11 (uniform, std 2^-11/sqrt(3) each) give an error std of
about 4.9e-4 of the output's RMS, and 3e-3 is six of those.  (Without decay
the state grows like the square root of the tokens summed: measured on GB300,
1024 decay-free tokens already put 63 of 524288 outputs past the elementwise
bound, by at most 0.017 against 0.0107.)  final_state keeps the elementwise
bound everywhere (its own relative error is ~2^-11), and dt = 0 keeps the state
at its initial size, so those use the elementwise bound.
"""
import numpy as np
import pytest
import torch

import oracle
from state_space_sequence_ssd_gb300 import _ffi
from state_space_sequence_ssd_gb300 import inputs as I

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 1e-2


@pytest.fixture(scope="module")
def ssd():
    from state_space_sequence_ssd_gb300 import build
    build.build()
    import state_space_sequence_ssd_gb300 as m
    m.ssd_get_device_error()  # start from clear error words
    return m


NORMWISE = 3e-3  # float16 operand rounding relative to the output's scale (see the module docstring)


def assert_close(name, got, ref, atol=ATOL, rtol=RTOL, normwise=0.0):
    """Elementwise comparison; with `normwise`, the bound also grows by normwise * the RMS of ref over each
    (batch, head) unit (axis 0 of the unit-stacked arrays)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    if normwise:
        rms = np.sqrt(np.mean(ref.reshape(ref.shape[0], -1) ** 2, axis=1))
        bound = bound + normwise * rms.reshape((-1,) + (1,) * (ref.ndim - 1))
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"got {got[i]} ref {ref[i]} err {err[i]} bound {bound[i]}")


def sample_units(w, k, seed=0):
    """k (batch, head) units including the first and last, and the first head of every group."""
    n = w.batch * w.nheads
    if k >= n:
        return np.arange(n)
    hpg = w.nheads // w.ngroups
    u = {0, n - 1} | {g * hpg for g in range(w.ngroups)}
    rng = np.random.default_rng(seed)
    while len(u) < k:
        u.add(int(rng.integers(0, n)))
    return np.array(sorted(u))


def rows(t, w, units):
    t = t.float().cpu().numpy()
    return np.stack([t[u // w.nheads, :, u % w.nheads] for u in units])


def states(t, w, units):
    t = t.cpu().numpy()
    return np.stack([t[u // w.nheads, u % w.nheads] for u in units])


def run(ssd, w, inp):
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    y, fin = ssd.ssd_forward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], w.chunk_size)
    torch.cuda.synchronize()
    return y, fin, ssd.ssd_get_device_error()


def oracle_ref(w, inp, units):
    n = I.as_numpy(inp)
    return oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], w.chunk_size, units=units)


# ------------------------------------------------------------------ A = 0: the jump formula


@pytest.mark.parametrize("N", [128, 256])
def test_no_decay_is_the_jump_formula(ssd, N):
    w = I.Workload("nodecay", 1, 16384, 8, 64, N, 2, 256, True)
    inp = I.make_inputs(w, seed=31)
    inp["A"] = torch.zeros_like(inp["A"])
    y, fin, st = run(ssd, w, inp)
    assert st == 0, f"device status {st}"
    units = sample_units(w, 4, seed=N)
    # the jump formula over the whole sequence: final = init + X^T diag(dt) B, per (batch, head)
    x = inp["x"].double().numpy()
    B = inp["B"].double().numpy()
    dt = inp["dt"].double().numpy()
    init = inp["init"].double().numpy()
    hpg = w.nheads // w.ngroups
    jump = np.stack([init[u // w.nheads, u % w.nheads]
                     + (x[u // w.nheads, :, u % w.nheads, :] * dt[u // w.nheads, :, u % w.nheads, None]).T
                     @ B[u // w.nheads, :, (u % w.nheads) // hpg, :] for u in units])
    assert_close("final vs jump formula", states(fin, w, units), jump)
    ref = oracle_ref(w, inp, units)
    assert_close("y", rows(y, w, units), ref["y"], normwise=NORMWISE)
    assert_close("final", states(fin, w, units), ref["final"])


# ------------------------------------------------------------------ dt = 0


def test_zero_dt_chunk_and_last_token(ssd):
    w = I.Workload("zerodt", 1, 4096 + 37, 8, 64, 128, 2, 256, True)
    inp = I.make_inputs(w, seed=32)
    inp["dt"][:, 3 * 256:4 * 256, :] = 0.0   # a whole chunk: no decay, no input
    inp["dt"][:, -1, :] = 0.0                # the last token of the ragged tail
    y, fin, st = run(ssd, w, inp)
    assert st == 0, f"device status {st}"
    units = np.arange(w.batch * w.nheads)
    ref = oracle_ref(w, inp, units)
    assert_close("y", rows(y, w, units), ref["y"])
    assert_close("final", states(fin, w, units), ref["final"])


@pytest.mark.parametrize("N,Q", [(64, 64), (256, 128)])
def test_zero_dt_everywhere_keeps_the_state(ssd, N, Q):
    """dt = 0: the state never moves, so final = init and y_t = C_t . init + D x_t (closed form)."""
    w = I.Workload("dt0", 1, 1000, 4, 64, N, 2, Q, True)
    inp = I.make_inputs(w, seed=33)
    inp["dt"] = torch.zeros_like(inp["dt"])
    y, fin, st = run(ssd, w, inp)
    assert st == 0, f"device status {st}"
    assert torch.equal(fin.cpu(), inp["init"]), "final_state must equal init_state exactly"
    x = inp["x"].double().numpy()[0]          # (L, H, P)
    C = inp["C"].double().numpy()[0]          # (L, G, N)
    init = inp["init"].double().numpy()[0]    # (H, P, N)
    D = inp["D"].double().numpy()
    hpg = w.nheads // w.ngroups
    want = np.stack([C[:, h // hpg, :] @ init[h].T + D[h] * x[:, h, :] for h in range(w.nheads)], axis=1)
    assert_close("y", y[0].float().cpu().numpy(), want)


# ------------------------------------------------------------------ float16 range


@pytest.mark.parametrize("absA", [1e-3, 1.0])
@pytest.mark.parametrize("scale", [8, 64, 256])
def test_magnitude_sweep_matches_or_reports_range(ssd, scale, absA):
    w = I.Workload("mag", 1, 4096, 8, 64, 128, 1, 256, True)
    inp = I.make_inputs(w, seed=34)
    for k in ("x", "B", "C"):  # powers of two: the bfloat16 inputs scale exactly
        inp[k] = (inp[k].float() * scale).to(torch.bfloat16)
    inp["A"] = torch.full_like(inp["A"], -absA)
    y, fin, st = run(ssd, w, inp)
    assert st in (0, _ffi.SSD_ERR_RANGE), f"device status {st}"
    if scale == 8:
        assert st == 0, "inputs of magnitude ~8 stay well inside float16's range"
    if scale == 256:
        assert st == _ffi.SSD_ERR_RANGE, "inputs of magnitude ~256 push the masked matrix past 65504"
    if st == 0:
        units = np.arange(w.batch * w.nheads)
        ref = oracle_ref(w, inp, units)
        assert_close(f"y x{scale} |A|={absA}", rows(y, w, units), ref["y"], normwise=NORMWISE)
        assert_close(f"final x{scale} |A|={absA}", states(fin, w, units), ref["final"], normwise=NORMWISE)


def test_range_flag_clears_after_a_read(ssd):
    """A call past float16's range reports SSD_ERR_RANGE once; the next in-range call is clean and right."""
    w = I.Workload("mag", 1, 512, 4, 64, 64, 1, 64, False)
    inp = I.make_inputs(w, seed=35)
    big = dict(inp)
    big["x"] = (inp["x"].float() * 2.0 ** 17).to(torch.bfloat16)  # x itself beyond 65504
    _, _, st = run(ssd, w, big)
    assert st == _ffi.SSD_ERR_RANGE
    y, fin, st = run(ssd, w, inp)
    assert st == 0
    units = np.arange(w.nheads)
    ref = oracle_ref(w, inp, units)
    assert_close("y", rows(y, w, units), ref["y"])
