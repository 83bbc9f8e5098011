"""GPU parity of ssd_backward against the fp64 oracle's reverse mode.

The oracle (``oracle.backward``) is the adjoint of the token recurrence,
pinned in test_oracle_backward_pins.py against the forward definition.  The
kernels compute the same gradients in the chunked form with float16 operands
and float32 accumulation (one rounding of each derived operand: the masked
matrices, the scaled x and dy rows, the block-start states and gradients).

Tolerances.  Each gradient is a sum of products (an inner product over the
state, over a group's heads, over tokens): dx_t = dt_t sum_n B_t[n] lam_t[n] +
D dy_t, ddt_t = A exp(dt_t A) <lam_t, state_{t-1}> + <lam_t, B_t x_t^T>, and
so on.  The kernels round the factors of those products to float16 (relative
error <= u = 2^-11 each, two factors per product) and accumulate in float32,
so the error of a computed gradient is bounded by about 2u times S, the sum of
the magnitudes of its products -- the usual componentwise bound of an inner
product -- and not by its value, which can be far smaller where the products
cancel (<lam, state> over 8192 state entries is the typical case).  The
oracle returns S for every gradient (``oracle.backward_terms``), and every
element is checked against

    |err| <= 1e-2 + 1e-2 |ref| + 2^-9 S        (2^-9 = 4u: two roundings, doubled)

With a single product S = |ref|, and the bound is the forward's elementwise
1e-2 + 1e-2 |ref| up to 0.2%.
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
    m.ssd_get_device_error()
    return m


SCALE_RTOL = 2.0 ** -9


def check(name, got, ref, scale=None):
    """|got - ref| <= ATOL + RTOL |ref| + 2^-9 scale elementwise (scale: the sum of the magnitudes of the
    products the gradient adds up)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    if scale is not None:
        bound = bound + SCALE_RTOL * np.asarray(scale, np.float64)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"got {got[i]} ref {ref[i]} err {err[i]} bound {bound[i]}")
    return float(np.max(err / bound))


def run_gpu(ssd, inp, gr, chunk_size):
    d = {k: (None if v is None else v.cuda()) for k, v in {**inp, **gr}.items()}
    out = ssd.ssd_backward(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["init"], d["dy"], d["dfinal"],
                           chunk_size=chunk_size)
    torch.cuda.synchronize()
    st = ssd.ssd_get_device_error()
    return {k: (None if v is None else v.float().cpu().numpy()) for k, v in out.items()}, st


def run_oracle(inp, gr):
    n = I.as_numpy(inp)
    g = I.as_numpy(gr)
    return oracle.backward_terms(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], g["dy"], g["dfinal"])


def compare_all(got, ref):
    for k in ("dx", "ddt", "dB", "dC", "dA", "dD", "dinit"):
        check(k, got[k], ref[k], ref["scales"][k])


CASES = [
    # name, batch, L, H, P, N, G, chunk, init, dfinal
    ("tiny_N64", 1, 512, 4, 64, 64, 1, 64, False, False),
    ("ragged_N128_G2", 2, 1000, 4, 64, 128, 2, 256, True, True),
    ("one_token", 1, 1, 2, 64, 64, 1, 64, True, True),
    ("ragged_N64_G4", 1, 700, 8, 64, 64, 4, 128, True, False),
    ("block_edge_N128", 1, 256, 4, 64, 128, 1, 128, False, True),
    ("groups_eq_heads", 1, 600, 4, 64, 64, 4, 64, True, True),  # one head per group: no cluster split
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(ssd, case):
    name, b, L, H, P, N, G, Q, init, dfin = case
    w = I.Workload(name, b, L, H, P, N, G, Q, init)
    inp = I.make_inputs(w, seed=51)
    gr = I.make_grad_inputs(w, seed=51, dfinal=dfin)
    got, st = run_gpu(ssd, inp, gr, Q)
    assert st == 0, f"device status {st}"
    ref = run_oracle(inp, gr)
    compare_all(got, ref)


def test_backward_without_D(ssd):
    w = I.Workload("noD", 1, 640, 4, 64, 128, 1, 256, True)
    inp = I.make_inputs(w, seed=52)
    inp["D"] = None
    gr = I.make_grad_inputs(w, seed=52)
    got, st = run_gpu(ssd, inp, gr, 256)
    assert st == 0
    ref = run_oracle(inp, gr)
    compare_all(got, ref)


def test_backward_chunk_size_does_not_matter(ssd):
    """The gradients do not depend on chunk_size (the kernels use their own blocks): bit-identical."""
    w = I.Workload("cs", 1, 1500, 4, 64, 64, 2, 64, True)
    inp = I.make_inputs(w, seed=53)
    gr = I.make_grad_inputs(w, seed=53)
    a, _ = run_gpu(ssd, inp, gr, 64)
    b_, _ = run_gpu(ssd, inp, gr, 256)
    for k in a:
        np.testing.assert_array_equal(a[k], b_[k], err_msg=k)


def test_backward_is_deterministic(ssd):
    w = I.WORKLOADS["mamba2_1p3b_layer_2x4096_N128"]
    inp = I.make_inputs(w, seed=54)
    gr = I.make_grad_inputs(w, seed=54)
    a, _ = run_gpu(ssd, inp, gr, w.chunk_size)
    b_, _ = run_gpu(ssd, inp, gr, w.chunk_size)
    for k in a:
        np.testing.assert_array_equal(a[k], b_[k], err_msg=k)


def test_backward_1p3b_layer(ssd):
    """2 x 4096 tokens, 64 heads, N 128: every output against the oracle over all 128 units."""
    w = I.WORKLOADS["mamba2_1p3b_layer_2x4096_N128"]
    inp = I.make_inputs(w, seed=55)
    gr = I.make_grad_inputs(w, seed=55)
    got, st = run_gpu(ssd, inp, gr, w.chunk_size)
    assert st == 0
    ref = run_oracle(inp, gr)
    compare_all(got, ref)


def test_backward_long_L65536_sparse_heads(ssd):
    """The full-size headline shape (1 x 65536, H 32, N 128, nonzero init) in the launch configuration the
    benchmark times.  dy and dfinal are non-zero on four heads only, so every group gradient (dB, dC)
    is the sum over those four heads and the oracle needs only their four units; the kernels still
    walk all 32 heads."""
    w = I.WORKLOADS["long_L65536_N128"]
    inp = I.make_inputs(w, seed=56)
    gr = I.make_grad_inputs(w, seed=56)
    active = [0, 9, 22, 31]
    mask = torch.zeros(w.nheads, dtype=torch.bool)
    mask[active] = True
    gr["dy"] = torch.where(mask[None, None, :, None], gr["dy"].float(), 0.0).to(torch.bfloat16)
    gr["dfinal"] = torch.where(mask[None, :, None, None], gr["dfinal"], 0.0)
    got, st = run_gpu(ssd, inp, gr, w.chunk_size)
    assert st == 0
    n = I.as_numpy(inp)
    g = I.as_numpy(gr)
    r = oracle.backward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], g["dy"], g["dfinal"],
                        units=active, scales=True)
    for i, h in enumerate(active):
        check(f"dx h{h}", got["dx"][0, :, h], r["dx"][i], r["dx_s"][i])
        check(f"ddt h{h}", got["ddt"][0, :, h], r["ddt"][i], r["ddt_s"][i])
        check(f"dinit h{h}", got["dinit"][0, h], r["dinit"][i], r["dinit_s"][i])
        check(f"dA h{h}", got["dA"][h], r["dA"][i], r["dA_s"][i])
        check(f"dD h{h}", got["dD"][h], r["dD"][i], r["dD_s"][i])
    check("dB", got["dB"][0, :, 0], r["dB"].sum(axis=0), r["dB_s"].sum(axis=0))
    check("dC", got["dC"][0, :, 0], r["dC"].sum(axis=0), r["dC_s"].sum(axis=0))
    # heads with no incoming gradient: zero dx; dA of those heads is zero too
    quiet = [h for h in range(w.nheads) if h not in active]
    assert np.all(got["dx"][0, :, quiet] == 0)
    assert np.all(got["dA"][quiet] == 0)


def test_backward_slow_decay(ssd):
    """|A| in [0.001, 0.01]: the state and the gradient into it carry over all 32 blocks, so every block
    start adds up many earlier blocks' terms (which the hops read as float16) -- the regime where their
    rounding adds up most."""
    w = I.Workload("slow", 1, 4096, 4, 64, 128, 1, 128, True)
    inp = I.make_inputs(w, seed=58)
    g = torch.Generator().manual_seed(58)
    inp["A"] = -(0.001 + 0.009 * torch.rand((w.nheads,), generator=g))
    gr = I.make_grad_inputs(w, seed=58)
    got, st = run_gpu(ssd, inp, gr, 128)
    assert st == 0
    ref = run_oracle(inp, gr)
    compare_all(got, ref)


def test_backward_rejects_unsupported(ssd):
    w = I.Workload("n256", 1, 256, 4, 64, 256, 1, 256, False)
    inp = I.make_inputs(w, seed=57)
    gr = I.make_grad_inputs(w, seed=57)
    with pytest.raises(ssd.SSDError) as e:
        run_gpu(ssd, inp, gr, 256)
    assert e.value.status == _ffi.SSD_ERR_UNSUPPORTED
