"""Pins for the CPU oracle (no GPU): the C recurrence against closed forms,
a hand-worked example, invariants and special cases.

Each pin is chosen so that a plausible slip in the oracle (a dropped dt, a
wrong decay index, an exclusive instead of inclusive cumsum, a transposed
state, a wrong head-to-group map) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import closed_form as cf
from state_space_sequence_ssd_gb300.inputs import Workload, as_numpy, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(L=37, H=4, P=8, N=6, G=2, Q=16, b=2, init=True, seed=1):
    w = Workload("pin", b, L, H, P, N, G, Q, init)
    return w, as_numpy(make_inputs(w, seed))


def _bits(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _run(i, Q):
    return oracle.forward(i["x"], i["dt"], i["A"], i["B"], i["C"], i["D"], i["init"], Q,
                          want_chunk_starts=True)


def _by_unit(o, b, H):
    """(nunits, ...) oracle output for all units -> (b, H, ...)."""
    return o.reshape((b, H) + o.shape[1:])


def test_golden_hand_example():
    """Hand-worked two-head example (tests/golden/hand_two_heads.json)."""
    g = json.load(open(os.path.join(GOLDEN, "hand_two_heads.json")))
    d = g["dims"]
    x, B, C = _bits(g["x"]), _bits(g["B"]), _bits(g["C"])
    dt = np.array(g["dt"], np.float32)
    A = np.array(g["A"], np.float32)
    D = np.array(g["D"], np.float32)
    o = oracle.forward(x, dt, A, B, C, D, None, d["chunk_size"])
    y = _by_unit(o["y"], 1, 2).transpose(0, 2, 1, 3)          # (b, L, H, P)
    np.testing.assert_allclose(y, np.array(g["expected_y"]), atol=g["tolerance"])
    np.testing.assert_allclose(o["final"].reshape(1, 2, 2, 2), np.array(g["expected_final"]),
                               atol=g["tolerance"])
    cs, _ = oracle.dA_cumsum(dt, A, d["chunk_size"])
    np.testing.assert_allclose(cs[0, 1, 0], g["expected_dA_cumsum_head1"], atol=1e-7)


@pytest.mark.parametrize("L,H,G,init", [(1, 2, 1, True), (5, 2, 2, False), (9, 4, 2, True), (16, 3, 1, True)])
def test_brute_force_quadratic_form(L, H, G, init):
    """P2: recurrence == literal unrolled sum over source tokens, tiny L."""
    w, i = _small(L=L, H=H, G=G, P=3, N=4, Q=4, b=1, init=init, seed=L)
    o = _run(i, 4)
    yq, fq = cf.quadratic_form(i["x"], i["dt"], i["A"], i["B"], i["C"], i["D"], i["init"])
    y = _by_unit(o["y"], 1, H).transpose(0, 2, 1, 3)
    np.testing.assert_allclose(y, yq, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(_by_unit(o["final"], 1, H), fq, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("Q", [4, 16, 64])
def test_chunked_closed_form(Q):
    """P3: recurrence == naive chunked form (segsum, chunk states, hop), ragged last chunk."""
    w, i = _small(L=75, Q=Q)
    o = _run(i, Q)
    yc, fc, sc, Sc = cf.chunked_form(i["x"], i["dt"], i["A"], i["B"], i["C"], i["D"], i["init"], Q)
    y = _by_unit(o["y"], w.batch, w.nheads).transpose(0, 2, 1, 3)
    np.testing.assert_allclose(y, yc, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(_by_unit(o["final"], w.batch, w.nheads), fc, rtol=1e-10, atol=1e-11)
    starts = _by_unit(o["chunk_starts"], w.batch, w.nheads).transpose(0, 2, 1, 3, 4)
    np.testing.assert_allclose(starts, sc, rtol=1e-10, atol=1e-11)
    S = oracle.chunk_states(i["x"], i["dt"], i["A"], i["B"], Q)
    S = _by_unit(S, w.batch, w.nheads).transpose(0, 2, 1, 3, 4)
    np.testing.assert_allclose(S, Sc, rtol=1e-10, atol=1e-11)


def test_jump_formula_without_decay():
    """P1: A = 0 -> final = init + B^T (dt X), a single matrix product (the jump formula)."""
    w, i = _small(L=50, Q=16)
    i["A"] = np.zeros_like(i["A"])
    o = _run(i, 16)
    yj, fj = cf.jump_formula_no_decay(i["x"], i["dt"], i["B"], i["C"], i["D"], i["init"])
    np.testing.assert_allclose(_by_unit(o["final"], w.batch, w.nheads), fj, rtol=1e-12, atol=1e-12)
    y = _by_unit(o["y"], w.batch, w.nheads).transpose(0, 2, 1, 3)
    np.testing.assert_allclose(y, yj, rtol=1e-11, atol=1e-11)


def test_split_sequence_resume():
    """P5: running [0, L1) then [L1, L) from the first final state equals one run."""
    w, i = _small(L=64, Q=16)
    o = _run(i, 16)
    L1 = 23
    first = {k: (v[:, :L1].copy() if k in ("x", "dt", "B", "C") else v) for k, v in i.items()}
    second = {k: (v[:, L1:].copy() if k in ("x", "dt", "B", "C") else v) for k, v in i.items()}
    o1 = _run(first, 16)
    second["init"] = o1["final"].reshape(w.batch, w.nheads, w.headdim, w.dstate).astype(np.float32)
    # the handoff goes through float32; compare against a run whose init is the same float32 rounding
    o2 = _run(second, 16)
    np.testing.assert_allclose(o2["final"], o["final"], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(o1["y"], o["y"][:, :L1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o2["y"], o["y"][:, L1:], rtol=1e-5, atol=1e-5)


def test_zero_dt_keeps_state():
    """P6: dt = 0 -> y = C . init + D x and final = init."""
    w, i = _small(L=20, Q=8)
    i["dt"] = np.zeros_like(i["dt"])
    o = _run(i, 8)
    np.testing.assert_allclose(o["final"].reshape(i["init"].shape), i["init"], rtol=0, atol=0)
    x = cf.bf16_bits_to_f64(i["x"])
    C = cf.bf16_bits_to_f64(i["C"])
    H, G = w.nheads, w.ngroups
    for b in range(w.batch):
        for h in range(H):
            g = h // (H // G)
            exp = C[b, :, g] @ i["init"][b, h].astype(np.float64).T + i["D"][h] * x[b, :, h]
            np.testing.assert_allclose(o["y"][b * H + h], exp, rtol=1e-12, atol=1e-12)


def test_single_token_closed_form():
    """P6: L = 1 -> h = e^{dt A} init + dt B x^T."""
    w, i = _small(L=1, Q=4)
    o = _run(i, 4)
    x, B = cf.bf16_bits_to_f64(i["x"]), cf.bf16_bits_to_f64(i["B"])
    H, G = w.nheads, w.ngroups
    for b in range(w.batch):
        for h in range(H):
            g = h // (H // G)
            dt = float(i["dt"][b, 0, h])
            hs = math.exp(dt * float(i["A"][h])) * i["init"][b, h].astype(np.float64) \
                + dt * np.outer(x[b, 0, h], B[b, 0, g])
            np.testing.assert_allclose(o["final"][b * H + h], hs, rtol=1e-13, atol=1e-14)


def test_memoryless_limit():
    """P6: huge |A| dt -> the state forgets everything but the current token."""
    w, i = _small(L=30, Q=8, init=True)
    i["A"] = np.full_like(i["A"], -1.0e4)
    i["dt"] = np.maximum(i["dt"], np.float32(0.05))
    o = _run(i, 8)
    x, B, C = (cf.bf16_bits_to_f64(i[k]) for k in ("x", "B", "C"))
    H, G = w.nheads, w.ngroups
    for b in range(w.batch):
        for h in range(H):
            g = h // (H // G)
            dt = i["dt"][b, :, h].astype(np.float64)
            exp = (np.sum(C[b, :, g] * B[b, :, g], axis=1) * dt)[:, None] * x[b, :, h] + i["D"][h] * x[b, :, h]
            np.testing.assert_allclose(o["y"][b * H + h], exp, rtol=1e-12, atol=1e-12)


def test_linearity_in_x_and_init():
    """P6: y and final are linear in (x, init) (values chosen so bf16 sums are exact)."""
    w, i = _small(L=21, Q=8)
    rng = np.random.default_rng(0)
    xa = rng.integers(-4, 5, size=i["x"].shape).astype(np.float32) / 4
    xb = rng.integers(-4, 5, size=i["x"].shape).astype(np.float32) / 4
    ia = (rng.integers(-4, 5, size=i["init"].shape) / 8).astype(np.float32)
    ib = (rng.integers(-4, 5, size=i["init"].shape) / 8).astype(np.float32)
    runs = []
    for xv, iv in ((xa, ia), (xb, ib), (xa + 2 * xb, ia + 2 * ib)):
        j = dict(i, x=_bits(xv), init=iv)
        runs.append(_run(j, 8))
    for k in ("y", "final"):
        np.testing.assert_allclose(runs[2][k], runs[0][k] + 2 * runs[1][k], rtol=1e-12, atol=1e-12)


def test_groups_replicated_equal_single_group():
    """P6: G = H with B/C replicated per head equals G = 1 (head-to-group mapping)."""
    w, i = _small(L=19, H=4, G=1, Q=8)
    o1 = _run(i, 8)
    j = dict(i, B=np.repeat(i["B"], 4, axis=2), C=np.repeat(i["C"], 4, axis=2))
    o4 = _run(j, 8)
    for k in ("y", "final"):
        np.testing.assert_array_equal(o1[k], o4[k])


def test_group_mapping_is_contiguous():
    """Heads [0, H/G) read group 0, the next H/G heads group 1, ...: perturbing group 1 moves only heads 2, 3."""
    w, i = _small(L=12, H=4, G=2, Q=4)
    o = _run(i, 4)
    B2 = i["B"].copy()
    B2[:, :, 1] = _bits(np.ones(B2[:, :, 1].shape, np.float32))
    o2 = _run(dict(i, B=B2), 4)
    y, y2 = _by_unit(o["y"], w.batch, 4), _by_unit(o2["y"], w.batch, 4)
    np.testing.assert_array_equal(y[:, :2], y2[:, :2])
    assert np.abs(y[:, 2:] - y2[:, 2:]).max() > 1e-3


def test_dA_cumsum_properties():
    """P7: last element = log2(e) A sum(dt); non-increasing; zero padding past L; dt_t layout."""
    w, i = _small(L=45, Q=16)
    cs, dtt = oracle.dA_cumsum(i["dt"], i["A"], 16)
    assert cs.shape == (w.batch, w.nheads, 3, 16)
    dt = i["dt"].astype(np.float64)
    for b in range(w.batch):
        for h in range(w.nheads):
            for c in range(3):
                seg = dt[b, c * 16:min(45, c * 16 + 16), h]
                exp = math.log2(math.e) * float(i["A"][h]) * math.fsum(seg)
                assert abs(cs[b, h, c, -1] - exp) <= 1e-12 * max(1.0, abs(exp))
                assert np.all(np.diff(cs[b, h, c]) <= 0)
                np.testing.assert_array_equal(dtt[b, h, c, :len(seg)], seg)
    # chunk 2 holds tokens 32..44: positions 13..15 are padding
    assert np.all(dtt[:, :, 2, 13:] == 0)
    assert np.all(cs[:, :, 2, 13:] == cs[:, :, 2, 12:13])
    # inclusive: the first element already holds token 0's term
    np.testing.assert_allclose(cs[:, :, :, 0], math.log2(math.e) * dtt[:, :, :, 0] * i["A"][None, :, None].astype(np.float64), rtol=1e-15)


def test_state_passing_reproduces_chunk_starts():
    """The chunk hop applied to per-chunk states reproduces the recurrence's chunk-start states."""
    w, i = _small(L=70, Q=16)
    o = _run(i, 16)
    S = oracle.chunk_states(i["x"], i["dt"], i["A"], i["B"], 16)
    S = _by_unit(S, w.batch, w.nheads).transpose(0, 2, 1, 3, 4)
    cs, _ = oracle.dA_cumsum(i["dt"], i["A"], 16)
    states, fin = oracle.state_passing(S.astype(np.float32), cs.astype(np.float32), i["init"], 16)
    starts = _by_unit(o["chunk_starts"], w.batch, w.nheads).transpose(0, 2, 1, 3, 4)
    # float32 rounding of the hop's inputs bounds the difference
    np.testing.assert_allclose(states, starts, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(fin, o["final"].reshape(fin.shape), rtol=1e-5, atol=1e-6)
    # states[0] is the initial state
    np.testing.assert_array_equal(states[:, 0], i["init"])


def test_chunk_scan_restarts_from_given_states():
    """compute_out oracle: restarting each chunk from the true chunk-start states reproduces y."""
    w, i = _small(L=50, Q=16)
    o = _run(i, 16)
    starts = _by_unit(o["chunk_starts"], w.batch, w.nheads).transpose(0, 2, 1, 3, 4).astype(np.float32)
    y = oracle.chunk_scan(i["x"], i["dt"], i["A"], i["B"], i["C"], i["D"], starts, 16)
    np.testing.assert_allclose(y, o["y"], rtol=1e-5, atol=1e-5)
    # and the same against the numpy chunked form
    yc, _, _, _ = cf.chunked_form(i["x"], i["dt"], i["A"], i["B"], i["C"], i["D"], i["init"], 16)
    np.testing.assert_allclose(y, yc.transpose(0, 2, 1, 3).reshape(y.shape), rtol=1e-5, atol=1e-5)


def test_unit_subset_matches_full_run():
    """Sampling (batch, head) units gives exactly the rows of a full run."""
    w, i = _small(L=33, Q=16)
    full = _run(i, 16)
    units = [5, 0, 7]
    sub = oracle.forward(i["x"], i["dt"], i["A"], i["B"], i["C"], i["D"], i["init"], 16, units=units)
    np.testing.assert_array_equal(sub["y"], full["y"][units])
    np.testing.assert_array_equal(sub["final"], full["final"][units])


# ---------------------------------------------------------------- input-side options
# dt_bias / softplus / clamp, D per channel and the z gate are not on the pages;
# the oracle takes their plainest reading.  Each pin ties one option to a
# different routine or a closed form (never to a retyped copy of itself).

def _f32_of_bits(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _plain(i, Q, **kw):
    a = dict(i)
    a.update(kw)
    return oracle.forward(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["init"], Q)


def test_options_that_change_nothing_reproduce_the_plain_path():
    w, i = _small(L=29, H=4, P=8, N=6, G=2)
    ref = _plain(i, 16)
    D2 = np.repeat(i["D"][:, None], w.headdim, axis=1)  # one weight per channel, equal to the head's
    o = oracle.forward(i["x"], i["dt"], i["A"], i["B"], i["C"], D2, i["init"], 16,
                       dt_bias=np.zeros(w.nheads, np.float32), dt_limit=(0.0, 1e30))
    np.testing.assert_array_equal(o["y"], ref["y"])
    np.testing.assert_array_equal(o["final"], ref["final"])


def test_softplus_and_bias_undo_their_inverse():
    """raw = log(expm1(d)) - bias: softplus(raw + bias) gives d back (numpy's expm1/log, not log1p/exp)."""
    w, i = _small(L=33, H=4, P=8, N=6, G=2)
    d = i["dt"].astype(np.float64)
    bias = (np.random.default_rng(3).standard_normal(w.nheads) * 0.5).astype(np.float32)
    raw = (np.log(np.expm1(d)) - bias.astype(np.float64)).astype(np.float32)
    o = oracle.forward(i["x"], raw, i["A"], i["B"], i["C"], i["D"], i["init"], 16,
                       dt_bias=bias, dt_softplus=True)
    ref = _plain(i, 16)
    np.testing.assert_allclose(o["y"], ref["y"], rtol=1e-4, atol=1e-7)
    np.testing.assert_allclose(o["final"], ref["final"], rtol=1e-4, atol=1e-7)
    # a large pre-activation passes through (softplus(v) -> v), a very negative one gives ~0
    big = np.full_like(i["dt"], 40.0)
    o2 = oracle.forward(i["x"], big, i["A"], i["B"], i["C"], i["D"], None, 16, dt_softplus=True)
    np.testing.assert_allclose(o2["y"], _plain(i, 16, dt=big, init=None)["y"], rtol=1e-12, atol=1e-14)
    o3 = oracle.forward(i["x"], np.full_like(i["dt"], -800.0), i["A"], i["B"], i["C"], i["D"], None, 16,
                        dt_softplus=True)
    np.testing.assert_allclose(o3["final"], 0.0, atol=1e-300)


def test_dt_limit_clamps_last():
    w, i = _small(L=40, H=4, P=8, N=6, G=2)
    d = i["dt"]
    lo, hi = np.float32(np.quantile(d, 0.25)), np.float32(np.quantile(d, 0.75))
    # equal bounds: a constant step
    o = oracle.forward(i["x"], d, i["A"], i["B"], i["C"], i["D"], i["init"], 16, dt_limit=(float(lo), float(lo)))
    ref = _plain(i, 16, dt=np.full_like(d, lo))
    np.testing.assert_allclose(o["y"], ref["y"], rtol=1e-12, atol=1e-14)
    # after the softplus, not before: softplus(log(expm1(d))) clamped equals d clamped
    raw = np.log(np.expm1(d.astype(np.float64))).astype(np.float32)
    o = oracle.forward(i["x"], raw, i["A"], i["B"], i["C"], i["D"], i["init"], 16, dt_softplus=True,
                       dt_limit=(float(lo), float(hi)))
    ref = _plain(i, 16, dt=np.clip(d, lo, hi))
    np.testing.assert_allclose(o["y"], ref["y"], rtol=1e-4, atol=1e-7)
    np.testing.assert_allclose(o["final"], ref["final"], rtol=1e-4, atol=1e-7)


def test_D_per_channel_closed_form():
    """With C = 0 the output is the skip term alone: y[b,t,h,p] = D[h,p] x[b,t,h,p] (H != P catches a transpose)."""
    w, i = _small(L=21, H=4, P=8, N=6, G=2)
    D2 = np.random.default_rng(5).standard_normal((w.nheads, w.headdim)).astype(np.float32)
    C0 = np.zeros_like(i["C"])
    o = oracle.forward(i["x"], i["dt"], i["A"], i["B"], C0, D2, i["init"], 16)
    y = _by_unit(o["y"], w.batch, w.nheads)                   # (b, H, L, P)
    x = _f32_of_bits(i["x"]).transpose(0, 2, 1, 3)            # (b, H, L, P)
    np.testing.assert_allclose(y, D2[None, :, None, :].astype(np.float64) * x, rtol=1e-15, atol=0)
    # and it adds to the state-space term exactly as the per-head weight does (linearity in D)
    ref0 = _plain(i, 16, D=None)
    o = oracle.forward(i["x"], i["dt"], i["A"], i["B"], i["C"], D2, i["init"], 16)
    np.testing.assert_allclose(_by_unit(o["y"] - ref0["y"], w.batch, w.nheads),
                               D2[None, :, None, :].astype(np.float64) * x, rtol=1e-12, atol=1e-12)


def test_z_gate_is_silu():
    """silu is pinned by two identities: g(z) - g(-z) = z and g(z) + g(-z) = z tanh(z/2)."""
    w, i = _small(L=25, H=4, P=8, N=6, G=2)
    y0 = _plain(i, 16)
    zf = np.random.default_rng(7).standard_normal(i["x"].shape).astype(np.float32) * 3
    z = _bits(zf)
    zneg = z ^ np.uint16(0x8000)                               # exact negation of a bf16 value
    op = oracle.forward(i["x"], i["dt"], i["A"], i["B"], i["C"], i["D"], i["init"], 16, z=z)
    on = oracle.forward(i["x"], i["dt"], i["A"], i["B"], i["C"], i["D"], i["init"], 16, z=zneg)
    zz = _f32_of_bits(z).transpose(0, 2, 1, 3).reshape(w.batch * w.nheads, w.seqlen, w.headdim)
    np.testing.assert_allclose(op["y"] - on["y"], zz * y0["y"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(op["y"] + on["y"], zz * np.tanh(zz / 2) * y0["y"], rtol=1e-12, atol=1e-13)
    # the gate touches the output only: the carried state is the ungated one
    np.testing.assert_array_equal(op["final"], y0["final"])
    oz = oracle.forward(i["x"], i["dt"], i["A"], i["B"], i["C"], i["D"], i["init"], 16, z=np.zeros_like(z))
    np.testing.assert_array_equal(oz["y"], 0.0)
