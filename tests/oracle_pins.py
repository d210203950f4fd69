"""Independent checks that pin the fp64 oracle to mathematics it must obey.

Each ``pin_*`` takes a recurrence callable with the signature of
``oracle.ssd_recurrence`` and raises ``AssertionError`` when the callable
disagrees with a result fixed by something other than the oracle itself:
the quadratic (dual) form of the SSD layer, a closed form, the impulse
response written as a product of per-step decays, the chunked algorithm
written out independently, or an algebraic invariant.

The same pins run against copies of the oracle with a planted mistake
(``test_oracle_mutants.py``) to show that every plausible slip fails one.
"""
from __future__ import annotations

import numpy as np

RTOL = 1e-11


def _rng(seed):
    return np.random.default_rng(seed)


def small_problem(seed, b=2, L=40, H=4, P=3, N=5, G=2, init=True, dt_scale=0.3):
    """Random fp64 problem with the Mamba-2 value ranges (A < 0, dt > 0).
    P != N so a transposed state is visible."""
    r = _rng(seed)
    x = r.standard_normal((b, L, H, P))
    dt = dt_scale * np.exp(r.uniform(np.log(0.05), np.log(2.0), (b, L, H)))
    A = -np.exp(r.uniform(0.0, np.log(16.0), H))
    B = r.standard_normal((b, L, G, N)) / np.sqrt(N)
    C = r.standard_normal((b, L, G, N)) / np.sqrt(N)
    D = r.standard_normal(H)
    s0 = 0.5 * r.standard_normal((b, H, P, N)) if init else None
    return x, dt, A, B, C, D, s0


def _close(got, want, rtol=RTOL, what=""):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    scale = max(np.max(np.abs(want)), 1e-300)
    err = np.max(np.abs(got - want)) if want.size else 0.0
    assert err <= rtol * scale, f"{what}: max|err|={err:.3e} scale={scale:.3e}"


# ---------------------------------------------------------------------------
# (p1) quadratic dual form
#   y = (L o C B^T)(dt o x) + D x + (exp(cum) o C) init,  L_ij = exp(sum_{k=j+1..i} dt_k A)
#   final = sum_j exp(cum_{L-1} - cum_j) dt_j x_j^T B_j + exp(cum_{L-1}) init
# ---------------------------------------------------------------------------
def quadratic_form(x, dt, A, B, C, D, s0):
    b, L, H, P = x.shape
    G = B.shape[2]
    N = B.shape[3]
    y = np.zeros_like(x)
    fin = np.zeros((b, H, P, N))
    for bi in range(b):
        for h in range(H):
            g = h * G // H
            cs = np.cumsum(dt[bi, :, h] * A[h])
            seg = cs[:, None] - cs[None, :]
            Lm = np.where(np.tril(np.ones((L, L), bool)), np.exp(np.minimum(seg, 0.0)), 0.0)
            CB = C[bi, :, g, :] @ B[bi, :, g, :].T
            u = dt[bi, :, h][:, None] * x[bi, :, h, :]
            yy = (Lm * CB) @ u
            if D is not None:
                yy += D[h] * x[bi, :, h, :]
            w = np.exp(cs[-1] - cs)
            ff = (w[:, None] * u).T @ B[bi, :, g, :]
            if s0 is not None:
                yy += np.exp(cs)[:, None] * (C[bi, :, g, :] @ s0[bi, h].T)
                ff += np.exp(cs[-1]) * s0[bi, h]
            y[bi, :, h, :] = yy
            fin[bi, h] = ff
    return y, fin


def pin_quadratic(rec):
    for seed, kw in ((1, {}), (2, dict(G=4)), (3, dict(G=1, init=False)), (4, dict(L=64, H=2, G=1, P=6, N=4))):
        x, dt, A, B, C, D, s0 = small_problem(seed, **kw)
        y, f = rec(x, dt, A, B, C, D, s0)
        yq, fq = quadratic_form(x, dt, A, B, C, D, s0)
        _close(y, yq, what="y vs quadratic form")
        _close(f, fq, what="final vs quadratic form")


# ---------------------------------------------------------------------------
# (p2) closed form, constant-decay scalar system
#   P = N = H = G = 1, dt = delta, A = alpha, B = C = x = 1, r = exp(delta alpha)
#   y_t = delta (1 - r^{t+1}) / (1 - r) + D + r^{t+1} h0
#   final = r^L h0 + delta (1 - r^L) / (1 - r)
# ---------------------------------------------------------------------------
def pin_closed_form(rec):
    for L, delta, alpha, d, h0 in ((37, 0.1, -2.0, 0.7, 1.5), (200, 0.013, -0.5, -1.1, -0.3), (5, 1.0, -16.0, 0.0, 2.0)):
        r = np.exp(delta * alpha)
        t = np.arange(L)
        want = delta * (1.0 - r ** (t + 1)) / (1.0 - r) + d + r ** (t + 1) * h0
        wantf = r ** L * h0 + delta * (1.0 - r ** L) / (1.0 - r)
        ones = np.ones((1, L, 1, 1))
        y, f = rec(ones, np.full((1, L, 1), delta), np.array([alpha]), ones, ones,
                   np.array([d]), np.full((1, 1, 1, 1), h0))
        _close(y[0, :, 0, 0], want, what="closed form y")
        _close(f.reshape(()), wantf, what="closed form final")


# ---------------------------------------------------------------------------
# (p3) impulse response: x = e_{t0} on one channel, zero init, no skip
#   y_t = (C_t . B_t0) dt_t0 prod_{k=t0+1..t} exp(dt_k A)   for t >= t0, else 0
# ---------------------------------------------------------------------------
def pin_impulse(rec):
    x, dt, A, B, C, D, _ = small_problem(5, b=1, L=30, H=2, P=2, N=4, G=1)
    for t0 in (0, 7, 29):
        for p in (0, 1):
            xi = np.zeros_like(x)
            xi[0, t0, :, p] = 1.0
            y, _ = rec(xi, dt, A, B, C, None, None)
            for h in range(2):
                want = np.zeros(30)
                decay = 1.0
                for t in range(t0, 30):
                    if t > t0:
                        decay *= np.exp(dt[0, t, h] * A[h])
                    want[t] = (C[0, t, 0] @ B[0, t0, 0]) * dt[0, t0, h] * decay
                _close(y[0, :, h, p], want, what=f"impulse t0={t0}")
                other = 1 - p
                assert np.all(y[0, :, h, other] == 0.0), "impulse leaked across channels"


# ---------------------------------------------------------------------------
# (p4) chunked SSD algorithm (written out here) == unchunked recurrence
#   for every chunk size, ragged last chunk included.
# ---------------------------------------------------------------------------
def chunked_form(x, dt, A, B, C, D, s0, Q):
    """The four SSD stages written out: in-chunk cumulative decay, chunk-local
    states, the sequential pass of states across chunks, and the chunk
    outputs (masked intra-chunk term + incoming-state term + skip).
    Returns y, final, and per (b, h) lists of the stage intermediates."""
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros_like(x)
    fin = np.zeros((b, H, P, N))
    nc = -(-L // Q)
    cums, locs, ins = {}, {}, {}
    for bi in range(b):
        for h in range(H):
            g = h * G // H
            hin = np.zeros((P, N)) if s0 is None else s0[bi, h].copy()
            for c in range(nc):
                s, e = c * Q, min(L, (c + 1) * Q)
                cs = np.cumsum(dt[bi, s:e, h] * A[h])                          # stage 1
                u = dt[bi, s:e, h][:, None] * x[bi, s:e, h, :]
                loc = (np.exp(cs[-1] - cs)[:, None] * u).T @ B[bi, s:e, g, :]   # stage 2
                Cc, Bc = C[bi, s:e, g, :], B[bi, s:e, g, :]
                seg = cs[:, None] - cs[None, :]
                Lm = np.where(np.tril(np.ones((e - s, e - s), bool)), np.exp(np.minimum(seg, 0.0)), 0.0)
                yy = (Lm * (Cc @ Bc.T)) @ u + np.exp(cs)[:, None] * (Cc @ hin.T)  # stage 4
                if D is not None:
                    yy += D[h] * x[bi, s:e, h, :]
                y[bi, s:e, h, :] = yy
                cums[bi, h, c], locs[bi, h, c], ins[bi, h, c] = cs, loc, hin.copy()
                hin = np.exp(cs[-1]) * hin + loc                                # stage 3
            fin[bi, h] = hin
    return y, fin, cums, locs, ins


def pin_chunked(rec):
    x, dt, A, B, C, D, s0 = small_problem(6, b=2, L=50, H=4, P=3, N=5, G=2)
    y0, f0 = rec(x, dt, A, B, C, D, s0)
    for Q in (1, 2, 7, 16, 25, 50, 64):
        y, f, *_ = chunked_form(x, dt, A, B, C, D, s0, Q)
        _close(y0, y, what=f"chunked Q={Q} y")
        _close(f0, f, what=f"chunked Q={Q} final")


# ---------------------------------------------------------------------------
# (p5) split / resume: run [0, L1) then [L1, L) from the returned state
# ---------------------------------------------------------------------------
def pin_split_resume(rec):
    x, dt, A, B, C, D, s0 = small_problem(7, L=45)
    y, f = rec(x, dt, A, B, C, D, s0)
    for L1 in (1, 17, 44):
        y1, f1 = rec(x[:, :L1], dt[:, :L1], A, B[:, :L1], C[:, :L1], D, s0)
        y2, f2 = rec(x[:, L1:], dt[:, L1:], A, B[:, L1:], C[:, L1:], D, f1)
        _close(np.concatenate([y1, y2], axis=1), y, what=f"split {L1} y")
        _close(f2, f, what=f"split {L1} final")


# ---------------------------------------------------------------------------
# (p6) linearity in x (zero init) and in the initial state (zero x)
# ---------------------------------------------------------------------------
def pin_linearity(rec):
    x1, dt, A, B, C, D, s1 = small_problem(8)
    x2, _, _, _, _, _, s2 = small_problem(9)
    a, c = 0.75, -1.25
    y1, f1 = rec(x1, dt, A, B, C, D, None)
    y2, f2 = rec(x2, dt, A, B, C, D, None)
    y, f = rec(a * x1 + c * x2, dt, A, B, C, D, None)
    _close(y, a * y1 + c * y2, what="linear in x: y")
    _close(f, a * f1 + c * f2, what="linear in x: final")
    z = np.zeros_like(x1)
    y1, f1 = rec(z, dt, A, B, C, D, s1)
    y2, f2 = rec(z, dt, A, B, C, D, s2)
    y, f = rec(z, dt, A, B, C, D, a * s1 + c * s2)
    _close(y, a * y1 + c * y2, what="linear in init: y")
    _close(f, a * f1 + c * f2, what="linear in init: final")


# ---------------------------------------------------------------------------
# (p7) dt = 0: nothing enters the state and nothing decays
# ---------------------------------------------------------------------------
def pin_dt_zero(rec):
    x, dt, A, B, C, D, s0 = small_problem(10)
    y, f = rec(x, np.zeros_like(dt), A, B, C, D, s0)
    G = B.shape[2]
    H = x.shape[2]
    want = D[None, None, :, None] * x
    for h in range(H):
        g = h * G // H
        want[:, :, h, :] += np.einsum("bln,bpn->blp", C[:, :, g, :], s0[:, h])
    _close(y, want, what="dt=0 y")
    _close(f, s0, what="dt=0 final")


# ---------------------------------------------------------------------------
# (p8) A -> 0: unnormalised causal linear attention
#   y_t = sum_{j<=t} (C_t . B_j) dt_j x_j + D x_t
# ---------------------------------------------------------------------------
def pin_linear_attention(rec):
    x, dt, A, B, C, D, _ = small_problem(11, G=1)
    A0 = np.full_like(A, -1e-13)
    y, _ = rec(x, dt, A0, B, C, D, None)
    L = x.shape[1]
    mask = np.tril(np.ones((L, L)))
    for bi in range(x.shape[0]):
        S = (C[bi, :, 0] @ B[bi, :, 0].T) * mask
        for h in range(x.shape[2]):
            want = S @ (dt[bi, :, h][:, None] * x[bi, :, h]) + D[h] * x[bi, :, h]
            _close(y[bi, :, h], want, rtol=1e-9, what="A->0 linear attention")


# ---------------------------------------------------------------------------
# (p9) groups: G groups equal the G = H run with B, C repeated per head
# ---------------------------------------------------------------------------
def pin_groups(rec):
    x, dt, A, B, C, D, s0 = small_problem(12, H=6, G=3)
    y, f = rec(x, dt, A, B, C, D, s0)
    rep = np.repeat(np.arange(3), 2)          # head h -> group h*G//H
    yr, fr = rec(x, dt, A, B[:, :, rep], C[:, :, rep], D, s0)
    _close(y, yr, what="grouped vs replicated y")
    _close(f, fr, what="grouped vs replicated final")
    # and a single head run on the group's B, C slice
    y1, f1 = rec(x[:, :, 5:6], dt[:, :, 5:6], A[5:6], B[:, :, 2:3], C[:, :, 2:3], D[5:6], s0[:, 5:6])
    _close(y1[:, :, 0], y[:, :, 5], what="head 5 alone")


# ---------------------------------------------------------------------------
# (p10) snapshots: the state entering chunk c equals the chunked algorithm's
#   passed state (stage 3), for several chunk sizes
# ---------------------------------------------------------------------------
def pin_snapshots(rec):
    x, dt, A, B, C, D, s0 = small_problem(13, b=2, L=48, H=4, P=3, N=5, G=2)
    for Q in (1, 5, 16, 48):
        _, f, _, _, ins = chunked_form(x, dt, A, B, C, D, s0, Q)
        y, f2, snaps = rec(x, dt, A, B, C, D, s0, snap_every=Q)
        for (bi, h, c), want in ins.items():
            _close(snaps[bi, c, h], want, what=f"snapshot Q={Q} chunk {c}")
        _close(f2, f, what="final with snapshots")


# ---------------------------------------------------------------------------
# (p11) in-chunk cumulative decay, entry by entry: for steps j <= i of chunk c
#   exp(cum[b,h,c,i] - cum[b,h,c,j]) = prod_{k=j+1..i} exp(dt_k A_h)
#   exp(cum[b,h,c,i])                = prod_{k=0..i}   exp(dt_k A_h)
# with k counted from the chunk's first step c*Q: the decay factors of the
# recurrence multiplied one step at a time (no running sum), so a permuted,
# mis-strided, exclusive or shifted layout inside a chunk fails here even
# when it keeps the chunk totals.
# ---------------------------------------------------------------------------
def pin_chunk_cumsum(fn):
    r = _rng(31)
    b, L, H = 2, 48, 3
    dt = 0.3 * np.exp(r.uniform(np.log(0.05), np.log(2.0), (b, L, H)))
    A = -np.exp(r.uniform(0.0, np.log(16.0), H))
    for Q in (1, 4, 16, 48):
        cum = np.asarray(fn(dt, A, Q))
        nc = L // Q
        assert cum.shape == (b, H, nc, Q), cum.shape
        for bi in range(b):
            for h in range(H):
                for c in range(nc):
                    dec = [np.exp(dt[bi, c * Q + k, h] * A[h]) for k in range(Q)]
                    for i in range(Q):
                        prod = 1.0
                        for k in range(i + 1):
                            prod *= dec[k]
                        _close(np.exp(cum[bi, h, c, i]), prod, rtol=1e-12, what=f"exp(cum) Q={Q} i={i}")
                        for j in range(i + 1):
                            pj = 1.0
                            for k in range(j + 1, i + 1):
                                pj *= dec[k]
                            _close(np.exp(cum[bi, h, c, i] - cum[bi, h, c, j]), pj, rtol=1e-12,
                                   what=f"exp(cum_i - cum_j) Q={Q} i={i} j={j}")


ALL_PINS = [pin_quadratic, pin_closed_form, pin_impulse, pin_chunked,
            pin_split_resume, pin_linearity, pin_dt_zero,
            pin_linear_attention, pin_groups, pin_snapshots]
