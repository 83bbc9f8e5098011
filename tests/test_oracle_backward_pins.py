"""Pins of the oracle's reverse mode (``oracle.backward``) against the forward definition.

The pages describe no backward pass; the oracle's is the adjoint of the
token recurrence.  These tests check it without trusting that derivation,
against the forward oracle itself (itself pinned in test_oracle_pins.py),
for the scalar loss

    Loss = sum(dy * y) + sum(dfinal * final)

* x, B, C, D and init enter Loss affinely (y and final are linear in each
  of them with the others fixed), so for ANY second value th' of one of
  them, Loss(th') - Loss(th) = <grad, th' - th> holds exactly in exact
  arithmetic: no step size, no truncation error.  B and C are shared by a
  group's heads, so their gradient is the sum of the heads' shares.
* dt and A enter through exp(dt A): central differences on values chosen
  exactly representable in float32 together with their perturbations, so
  the step is exact and only the O(step^2) truncation error remains.
* dy = 0: closed forms for dinit and dx (pure decay of dfinal), and for dinit's
  scale; with non-negative terms that scale equals dinit.
* The chunked algorithm (``closed_form.backward_chunked``), another route to
  the same numbers, agrees with the token recurrence for several blocks.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import closed_form as cf
from state_space_sequence_ssd_gb300 import inputs as I

W = I.Workload("bwd_pin", 2, 41, 4, 5, 6, 2, 16, True)


def draw(w=W, seed=5):
    n = I.as_numpy(I.make_inputs(w, seed=seed))
    g = I.as_numpy(I.make_grad_inputs(w, seed=seed))
    return n, g


def loss(n, g):
    H = n["x"].shape[2]
    b = n["x"].shape[0]
    r = oracle.forward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], 16)
    y = r["y"].reshape(b, H, *r["y"].shape[1:]).transpose(0, 2, 1, 3)
    fin = r["final"].reshape(b, H, *r["final"].shape[1:])
    dy = cf.bf16_bits_to_f64(g["dy"])
    val = np.sum(dy * y)
    if g["dfinal"] is not None:
        val += np.sum(g["dfinal"].astype(np.float64) * fin)
    return val


def grads(n, g):
    return oracle.backward_full(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], g["dy"], g["dfinal"])


def other_bf16(shape, seed):
    t = torch.randn(shape, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    return I.bf16_bits(t)


@pytest.mark.parametrize("name", ["x", "B", "C", "D", "init"])
def test_affine_inputs_exact_difference(name):
    n, g = draw()
    gr = grads(n, g)
    key = {"x": "dx", "B": "dB", "C": "dC", "D": "dD", "init": "dinit"}[name]
    m = dict(n)
    if n[name].dtype == np.uint16:
        m[name] = other_bf16(n[name].shape, 99)
        delta = cf.bf16_bits_to_f64(m[name]) - cf.bf16_bits_to_f64(n[name])
    else:
        rng = np.random.default_rng(7)
        m[name] = rng.standard_normal(n[name].shape).astype(np.float32)
        delta = m[name].astype(np.float64) - n[name].astype(np.float64)
    lhs = loss(m, g) - loss(n, g)
    rhs = np.sum(gr[key] * delta)
    scale = np.sum(np.abs(gr[key] * delta))
    assert abs(lhs - rhs) <= 1e-11 * scale, (name, lhs, rhs)


def exact_dt(w, seed):
    """dt = m 2^-12 (m in 1..255) and a perturbation of k 2^-26 (|k| <= 8): dt +- e exact in float32."""
    rng = np.random.default_rng(seed)
    dt = (rng.integers(1, 256, (w.batch, w.seqlen, w.nheads)) * 2.0 ** -12).astype(np.float32)
    e = rng.integers(-8, 9, dt.shape) * 2.0 ** -26
    assert np.all((dt.astype(np.float64) + e).astype(np.float32) == dt.astype(np.float64) + e)
    assert np.all((dt.astype(np.float64) - e).astype(np.float32) == dt.astype(np.float64) - e)
    return dt, e


def test_dt_central_difference():
    n, g = draw()
    n["dt"], e = exact_dt(W, 11)
    gr = grads(n, g)
    p, m = dict(n), dict(n)
    p["dt"] = (n["dt"].astype(np.float64) + e).astype(np.float32)
    m["dt"] = (n["dt"].astype(np.float64) - e).astype(np.float32)
    lhs = (loss(p, g) - loss(m, g)) / 2.0
    rhs = np.sum(gr["ddt"] * e)
    assert abs(lhs - rhs) <= 1e-6 * np.sum(np.abs(gr["ddt"] * e)), (lhs, rhs)


def test_dt_single_token_central_difference():
    """One token's dt alone: checks ddt at one position, not only along a random direction."""
    n, g = draw()
    n["dt"], _ = exact_dt(W, 12)
    gr = grads(n, g)
    for (bb, t, h) in [(0, 0, 0), (1, 20, 3), (0, 40, 2)]:
        e = 2.0 ** -22
        p, m = dict(n), dict(n)
        p["dt"] = n["dt"].copy(); p["dt"][bb, t, h] += e
        m["dt"] = n["dt"].copy(); m["dt"][bb, t, h] -= e
        lhs = (loss(p, g) - loss(m, g)) / (2 * e)
        assert abs(lhs - gr["ddt"][bb, t, h]) <= 1e-6 * (1 + abs(lhs)), (bb, t, h, lhs, gr["ddt"][bb, t, h])


def test_A_central_difference():
    n, g = draw()
    n["A"] = (-np.arange(1, W.nheads + 1) * 2.0 ** -3).astype(np.float32)  # -0.125 .. -0.5, exact
    gr = grads(n, g)
    for h in range(W.nheads):
        e = 2.0 ** -20
        p, m = dict(n), dict(n)
        p["A"] = n["A"].copy(); p["A"][h] += e
        m["A"] = n["A"].copy(); m["A"][h] -= e
        lhs = (loss(p, g) - loss(m, g)) / (2 * e)
        assert abs(lhs - gr["dA"][h]) <= 1e-6 * (1 + abs(lhs)), (h, lhs, gr["dA"][h])


def test_zero_dy_is_pure_decay_of_dfinal():
    """dy = 0: Loss = <dfinal, final>, so dinit = exp(A sum dt) dfinal and
    dx_s[p] = dt_s exp(A sum_{k>s} dt_k) sum_n B_s[n] dfinal[p][n] (closed forms)."""
    n, g = draw()
    g["dy"] = np.zeros_like(g["dy"])
    gr = grads(n, g)
    dt = n["dt"].astype(np.float64)
    A = n["A"].astype(np.float64)
    B = cf.bf16_bits_to_f64(n["B"])
    hpg = W.nheads // W.ngroups
    for bb in range(W.batch):
        for h in range(W.nheads):
            tot = np.exp(A[h] * dt[bb, :, h].sum())
            np.testing.assert_allclose(gr["dinit"][bb, h], tot * g["dfinal"][bb, h], rtol=1e-12, atol=1e-15)
            after = np.exp(A[h] * (dt[bb, :, h].sum() - np.cumsum(dt[bb, :, h])))  # sum over k > s
            want = (dt[bb, :, h] * after)[:, None] * (B[bb, :, h // hpg] @ g["dfinal"][bb, h].astype(np.float64).T)
            np.testing.assert_allclose(gr["dx"][bb, :, h], want, rtol=1e-11, atol=1e-14)
    assert np.all(gr["dC"] == 0) and gr["dD"].any() == False  # noqa: E712  (x . dy = 0 with dy = 0)


def terms(n, g):
    return oracle.backward_terms(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], g["dy"], g["dfinal"])


def test_dinit_scale_closed_forms():
    """dinit's scale (the magnitudes of the adjoint's terms C_t dy_t^T and dfinal, each decayed to the
    start):
    * dy = 0: one term, so it is exp(A sum dt) |dfinal|;
    * C, dy and dfinal >= 0: no term cancels, so it equals dinit (pinned above by exact differences);
    * otherwise it bounds |dinit| (triangle inequality) and exceeds it where the terms cancel."""
    n, g = draw()
    g0 = dict(g)
    g0["dy"] = np.zeros_like(g["dy"])
    r = terms(n, g0)
    dt = n["dt"].astype(np.float64)
    A = n["A"].astype(np.float64)
    for bb in range(W.batch):
        for h in range(W.nheads):
            tot = np.exp(A[h] * dt[bb, :, h].sum())
            np.testing.assert_allclose(r["scales"]["dinit"][bb, h], tot * np.abs(g["dfinal"][bb, h]), rtol=1e-12,
                                       atol=1e-15)
    npos, gpos = dict(n), dict(g)
    npos["C"] = n["C"] & np.uint16(0x7FFF)   # bf16 sign bit cleared: |C|
    gpos["dy"] = g["dy"] & np.uint16(0x7FFF)
    gpos["dfinal"] = np.abs(g["dfinal"])
    rp = terms(npos, gpos)
    np.testing.assert_allclose(rp["scales"]["dinit"], rp["dinit"], rtol=1e-12, atol=1e-15)
    r = terms(n, g)
    assert np.all(r["scales"]["dinit"] >= np.abs(r["dinit"]) * (1 - 1e-12))
    assert np.any(r["scales"]["dinit"] > 2 * np.abs(r["dinit"]))


def test_no_gradient_in_gives_zero():
    n, g = draw()
    g["dy"] = np.zeros_like(g["dy"])
    g["dfinal"] = None
    gr = grads(n, g)
    for k, v in gr.items():
        assert not np.any(v), k


@pytest.mark.parametrize("block", [1, 7, 16, 64])
def test_chunked_algorithm_matches_the_recurrence(block):
    w = W.with_(seqlen=53)
    n, g = draw(w, seed=9)
    r = grads(n, g)
    c = cf.backward_chunked(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], g["dy"], g["dfinal"], block)
    for k in r:
        np.testing.assert_allclose(c[k], r[k], rtol=1e-10, atol=1e-10 * np.max(np.abs(r[k])), err_msg=k)


def test_units_subset_matches_full():
    n, g = draw()
    full = oracle.backward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], g["dy"], g["dfinal"])
    sub = oracle.backward(n["x"], n["dt"], n["A"], n["B"], n["C"], n["D"], n["init"], g["dy"], g["dfinal"],
                          units=[1, 6])
    for k in full:
        np.testing.assert_array_equal(sub[k], full[k][[1, 6]], err_msg=k)
