"""numpy fp64 closed forms that pin the C recurrence -- TEST INFRASTRUCTURE ONLY.

Written independently of ``ssd_oracle.c`` (different route to the same
numbers), and used only by the CPU pin tests.  Citations by page title:

[disconfirmai] "Jane Street ML Engineers Map Mamba-2 Recurrent State
    Computation to Tensor Cores with cuTile": the three-kernel decomposition
    paragraph (chunk_cumsum / fwd_pass_state / compute_out with carried-state
    term, decayed causally masked interaction matrix and skip connection) and
    the jump-formula paragraph (h(t+T) = h(t) + B X^T with B, X the stacked
    per-token vectors; decay re-enters as log-space cumulative sums and row
    pre-scaling by exponentials).
[devotd] devotd.net page on the Mamba-2 cuTile forward kernels, sections 1-2.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _widen(x, dt, A, B, C, D, init):
    x = bf16_bits_to_f64(x)
    B = bf16_bits_to_f64(B)
    C = bf16_bits_to_f64(C) if C is not None else None
    dt = np.asarray(dt, np.float64)
    A = np.asarray(A, np.float64)
    b, L, H, P = x.shape
    N = B.shape[3]
    D = np.zeros(H) if D is None else np.asarray(D, np.float64)
    init = np.zeros((b, H, P, N)) if init is None else np.asarray(init, np.float64)
    return x, dt, A, B, C, D, init


def quadratic_form(x, dt, A, B, C, D, init):
    """Brute force, O(L^3) per head: the unrolled recurrence as a sum over source tokens.

    y_t = sum_{s<=t} (C_t . B_s) * prod_{s<k<=t} exp(dt_k A) * dt_s x_s
          + (C_t . h0) * prod_{k<=t} exp(dt_k A) + D x_t
    final = sum_s prod_{s<k<L} exp(dt_k A) dt_s B_s x_s^T + prod_k exp(dt_k A) h0
    Decay products are formed literally, one factor per token.  Small L only.
    Returns y (b, L, H, P) and final (b, H, P, N).
    """
    x, dt, A, B, C, D, init = _widen(x, dt, A, B, C, D, init)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros((b, L, H, P))
    fin = np.zeros((b, H, P, N))
    for bi in range(b):
        for h in range(H):
            g = h // (H // G)
            a = np.exp(dt[bi, :, h] * A[h])              # per-token decay factor
            h0 = init[bi, h].T                           # (N, P)
            for t in range(L):
                acc = np.zeros(P)
                for s in range(t + 1):
                    decay = 1.0
                    for k in range(s + 1, t + 1):
                        decay *= a[k]
                    acc += (C[bi, t, g] @ B[bi, s, g]) * decay * dt[bi, s, h] * x[bi, s, h]
                carry = 1.0
                for k in range(t + 1):
                    carry *= a[k]
                acc += carry * (C[bi, t, g] @ h0)
                y[bi, t, h] = acc + D[h] * x[bi, t, h]
            hs = np.zeros((N, P))
            for s in range(L):
                decay = 1.0
                for k in range(s + 1, L):
                    decay *= a[k]
                hs += decay * dt[bi, s, h] * np.outer(B[bi, s, g], x[bi, s, h])
            total = 1.0
            for k in range(L):
                total *= a[k]
            hs += total * h0
            fin[bi, h] = hs.T
    return y, fin


def chunked_form(x, dt, A, B, C, D, init, chunk_size):
    """Naive chunked closed form (the structure of the three kernels), fp64.

    Per chunk: cs = in-chunk inclusive cumsum of dt*A (natural log units);
      intra-chunk:   Y_diag = ((C B^T) * exp(cs_i - cs_j) [j<=i] * dt_j) X
      carried state: Y_off  = exp(cs_i) * (C h_c)
      chunk state:   S_c    = B^T (exp(cs_last - cs_j) dt_j X)      (jump formula with row pre-scaling)
      hop:           h_{c+1} = exp(cs_last) h_c + S_c
    Works for any chunk_size, including a ragged last chunk.
    Returns y (b, L, H, P), final (b, H, P, N), chunk_starts (b, nc, H, P, N), S (b, nc, H, P, N).
    """
    x, dt, A, B, C, D, init = _widen(x, dt, A, B, C, D, init)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    Q = chunk_size
    nc = -(-L // Q)
    y = np.zeros((b, L, H, P))
    fin = np.zeros((b, H, P, N))
    starts = np.zeros((b, nc, H, P, N))
    Sall = np.zeros((b, nc, H, P, N))
    for bi in range(b):
        for h in range(H):
            g = h // (H // G)
            hcur = init[bi, h].T.copy()                  # (N, P)
            for c in range(nc):
                t0, t1 = c * Q, min(L, (c + 1) * Q)
                Xc = x[bi, t0:t1, h]                     # (T, P)
                Bc = B[bi, t0:t1, g]                     # (T, N)
                Cc = C[bi, t0:t1, g]
                dtc = dt[bi, t0:t1, h]
                cs = np.cumsum(dtc * A[h])
                T = t1 - t0
                ii, jj = np.meshgrid(np.arange(T), np.arange(T), indexing="ij")
                mask = jj <= ii
                seg = np.where(mask, np.exp(np.where(mask, cs[:, None] - cs[None, :], 0.0)), 0.0)
                M = (Cc @ Bc.T) * seg * dtc[None, :]
                Yd = M @ Xc
                Yo = np.exp(cs)[:, None] * (Cc @ hcur)
                y[bi, t0:t1, h] = Yd + Yo + D[h] * Xc
                starts[bi, c, h] = hcur.T
                w = np.exp(cs[-1] - cs) * dtc
                S = Bc.T @ (w[:, None] * Xc)             # (N, P)
                Sall[bi, c, h] = S.T
                hcur = np.exp(cs[-1]) * hcur + S
            fin[bi, h] = hcur.T
    return y, fin, starts, Sall


def jump_formula_no_decay(x, dt, B, C, D, init):
    """A = 0: no decay, so the state after tokens [0, t] is h0 + B^T (dt * X) over those tokens.

    final = h0 + B^T (dt X)  -- one matrix product over the whole sequence, the
    jump formula h(t+T) = h(t) + B X^T with X pre-scaled by dt.
    y_t   = C_t . (h0 + sum_{s<=t} dt_s B_s x_s^T) + D x_t, via a running sum of outer products.
    """
    H = x.shape[2]
    A = np.zeros(H)
    x, dt, A, B, C, D, init = _widen(x, dt, A, B, C, D, init)
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros((b, L, H, P))
    fin = np.zeros((b, H, P, N))
    for bi in range(b):
        for h in range(H):
            g = h // (H // G)
            Xs = dt[bi, :, h, None] * x[bi, :, h]        # (L, P)
            Bg = B[bi, :, g]                             # (L, N)
            fin[bi, h] = (init[bi, h].T + Bg.T @ Xs).T
            outer = np.einsum("tn,tp->tnp", Bg, Xs)
            running = np.cumsum(outer, axis=0) + init[bi, h].T[None]
            y[bi, :, h] = np.einsum("tn,tnp->tp", C[bi, :, g], running) + D[h] * x[bi, :, h]
    return y, fin


def backward_chunked(x, dt, A, B, C, D, init, dy, dfinal, block):
    """Gradients by blocks of ``block`` tokens: the chunked reverse-mode algorithm, in numpy fp64.

    Per (batch, head) and block (c the inclusive cumulative sum of dt*A inside the block, c_e its
    last value, L[r, i] = exp(c_r - c_i) for r >= i, else 0; h0 the state before the block, mu the
    gradient flowing into the state after the block from later tokens):
        forward hop   h0_{k+1} = exp(c_e) h0_k + sum_j exp(c_e - c_j) dt_j B_j x_j^T
        backward hop  mu_{k-1} = exp(c_e) mu_k + sum_r exp(c_r) C_r dy_r^T,  mu_last = dfinal,
                      dinit = mu_{-1}
        G   = (L o C B^T)^T dY + diag(exp(c_e - c)) B mu        (lam_i^T B_i, rows i)
        dx  = diag(dt) G + D dY,   s_i = G_i . x_i
        Wd  = L o (dY X^T) o dt_j (columns j)
        dC  = diag(exp(c)) dY h0^T + Wd B      (this head's share)
        dB  = diag(dt exp(c_e - c)) X mu^T + Wd^T C
    and the gradient of the step log-decay l_t = dt_t A, split at the block's ends so that every sum
    stays inside the block (h0 reaching forward, mu reaching back, pairs of tokens inside the block):
        dl_t = exp(c_e) <mu, h0> + sum_{j<t} v_j + sum_{r>=t} (rho1_r + rho2_r - sigma_r),
        v_j = dt_j exp(c_e - c_j) x_j . (B mu)_j,   rho2_r = exp(c_r) dy_r . (C h0)_r,
        rho1_r = sum_j (Wd o C B^T)[r][j],          sigma_r = dt_r x_r . ((L o C B^T)^T dY)_r,
    so ddt_t = A dl_t + G_t . x_t and dA = sum_t dt_t dl_t.  Returns the layout of
    ``oracle.backward_full``.  Independent of the C oracle (same mathematics, different route).
    """
    x, dt, A, B, C, D, init = _widen(x, dt, A, B, C, D, init)
    dy = bf16_bits_to_f64(dy)
    b, L, H, P = x.shape
    G_, N = B.shape[2], B.shape[3]
    hpg = H // G_
    dfinal = np.zeros((b, H, P, N)) if dfinal is None else np.asarray(dfinal, np.float64)
    nblk = -(-L // block)
    out = {"dx": np.zeros((b, L, H, P)), "ddt": np.zeros((b, L, H)), "dB": np.zeros((b, L, G_, N)),
           "dC": np.zeros((b, L, G_, N)), "dA": np.zeros(H), "dD": np.zeros(H), "dinit": np.zeros((b, H, P, N))}
    for bb in range(b):
        for h in range(H):
            g = h // hpg
            blocks = [(k * block, min(L, (k + 1) * block)) for k in range(nblk)]
            cs = []
            for t0, t1 in blocks:
                cs.append(np.cumsum(dt[bb, t0:t1, h] * A[h]))
            # forward hop: state before each block (N x P)
            h0 = [init[bb, h].T.copy()]
            for k, (t0, t1) in enumerate(blocks[:-1]):
                c = cs[k]
                w = np.exp(c[-1] - c) * dt[bb, t0:t1, h]
                h0.append(np.exp(c[-1]) * h0[-1] + B[bb, t0:t1, g].T @ (w[:, None] * x[bb, t0:t1, h]))
            # backward hop: gradient into each block's final state
            mu = [None] * nblk
            cur = dfinal[bb, h].T.copy()
            for k in range(nblk - 1, -1, -1):
                t0, t1 = blocks[k]
                c = cs[k]
                mu[k] = cur
                cur = np.exp(c[-1]) * cur + C[bb, t0:t1, g].T @ (np.exp(c)[:, None] * dy[bb, t0:t1, h])
            dinit = cur
            out["dinit"][bb, h] = dinit.T
            for k, (t0, t1) in enumerate(blocks):
                c = cs[k]
                Lm = np.tril(np.exp(c[:, None] - c[None, :]))
                Xb, Yb = x[bb, t0:t1, h], dy[bb, t0:t1, h]
                Bb, Cb = B[bb, t0:t1, g], C[bb, t0:t1, g]
                dtb = dt[bb, t0:t1, h]
                ext = np.exp(c[-1] - c)
                CB = Cb @ Bb.T
                Gin = (Lm * CB).T @ Yb
                Gmu = Bb @ mu[k]
                Gm = Gin + ext[:, None] * Gmu
                out["dx"][bb, t0:t1, h] = dtb[:, None] * Gm + D[h] * Yb
                Wd = Lm * (Yb @ Xb.T) * dtb[None, :]
                out["dC"][bb, t0:t1, g] += np.exp(c)[:, None] * (Yb @ h0[k].T) + Wd @ Bb
                out["dB"][bb, t0:t1, g] += (dtb * ext)[:, None] * (Xb @ mu[k].T) + Wd.T @ Cb
                v = dtb * ext * np.sum(Xb * Gmu, axis=1)
                rho1 = np.sum(Wd * CB, axis=1)
                rho2 = np.exp(c) * np.sum(Yb * (Cb @ h0[k]), axis=1)
                sigma = dtb * np.sum(Xb * Gin, axis=1)
                w = rho1 + rho2 - sigma
                dl = (np.exp(c[-1]) * np.sum(mu[k] * h0[k]) + np.concatenate([[0.0], np.cumsum(v)[:-1]])
                      + np.cumsum(w[::-1])[::-1])
                out["ddt"][bb, t0:t1, h] = A[h] * dl + np.sum(Gm * Xb, axis=1)
                out["dA"][h] += np.sum(dtb * dl)
                out["dD"][h] += np.sum(Xb * Yb)
    return out
