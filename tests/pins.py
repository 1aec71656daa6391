"""Pins for the fp64 oracle: checks against facts the pages and the mathematics fix.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError if the oracle
disagrees. None of them re-types the oracle's loop: each uses a different route to
the same number (a printed worked example, a closed form, a convolution, explicit
products, a limit, an invariant). ``test_oracle_pins.py`` runs them on the real
oracle; ``test_oracle_mutants.py`` runs them on builds with one planted mistake each
and requires every mutant to fail at least one pin.
"""
from __future__ import annotations

import os

import numpy as np
from scipy.special import expit

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _silu(z):
    return z * expit(z)


def _softplus(r):
    return np.logaddexp(0.0, r)


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / scale)


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            vals[k] = [float(x) for x in v]
    return vals


def pin_worked_example(o):
    """'Mamba and State Space Models', 'A worked numerical pass': A = -1, step sizes
    0.1, 5.0, 0.1 give A-bar 0.905, 0.007, 0.905, and token 2 dominates the state."""
    g = _read_golden("worked_example.txt")
    A = np.array([[g["A"][0]]])
    delta = np.array(g["delta"]).reshape(1, 3, 1)
    # Decay only: start from h0 = 1 with zero input, so y_t = prod_{s<=t} A-bar_s.
    y, _ = o.selective_scan_fwd(np.zeros((1, 3, 1)), delta, A, np.ones((1, 3, 1)), np.ones((1, 3, 1)),
                                delta_softplus=False, h0=np.ones((1, 1, 1)))
    y = y.ravel()
    abar = [y[0], y[1] / y[0], y[2] / y[1]]
    assert [round(a, 3) for a in abar] == g["abar"], abar
    # Write-dominance: unit inputs at every token; token 2's share of h_3 exceeds 90%.
    y1, _ = o.selective_scan_fwd(np.ones((1, 3, 1)), delta, A, np.ones((1, 3, 1)), np.ones((1, 3, 1)),
                                 delta_softplus=False)
    share2 = abar[2] * g["delta"][1] / y1.ravel()[2]
    assert share2 > 0.9, share2


def pin_lti_convolution(o, seed=1):
    """Constant delta, B, C: y = K * u + D u with K_j = sum_n C_n exp(j dt A_n) dt B_n
    ("Arch 02: Mamba SSM" kernel K = (C B-bar, C A-bar B-bar, ...); "State Space Model
    (SSM)" glossary; "8.7 State Space Models (Mamba)" section 2.1), by brute force."""
    rng = np.random.default_rng(seed)
    b, L, D, N = 2, 37, 3, 5
    raw = rng.normal(-1.0, 0.7, (b, 1, D))
    bias = rng.normal(0.0, 0.3, D)
    A = -rng.uniform(0.2, 3.0, (D, N))
    B0 = rng.standard_normal((b, 1, N))
    C0 = rng.standard_normal((b, 1, N))
    u = rng.standard_normal((b, L, D))
    z = rng.standard_normal((b, L, D))
    Dk = rng.standard_normal(D)
    y, _ = o.selective_scan_fwd(u, np.repeat(raw, L, 1), A, np.repeat(B0, L, 1), np.repeat(C0, L, 1),
                                D=Dk, z=z, delta_bias=bias, delta_softplus=True)
    ref = np.zeros_like(y)
    for bi in range(b):
        for d in range(D):
            dt = _softplus(raw[bi, 0, d] + bias[d])
            j = np.arange(L)[:, None]
            K = (C0[bi, 0] * np.exp(j * dt * A[d]) * dt * B0[bi, 0]).sum(-1)  # (L,)
            for t in range(L):
                conv = np.dot(K[: t + 1][::-1], u[bi, : t + 1, d])
                ref[bi, t, d] = (conv + Dk[d] * u[bi, t, d]) * _silu(z[bi, t, d])
    assert _rel(y, ref) < 1e-11, _rel(y, ref)


def pin_delta_zero_holds_state(o, seed=2):
    """Delta -> 0 leaves the state untouched ("Arch 02: Mamba SSM": small Delta ~ pure
    copy; "Mamba and State Space Models": small Delta leaves the state untouched)."""
    rng = np.random.default_rng(seed)
    b, L, D, N = 2, 9, 4, 8
    u = rng.standard_normal((b, L, D))
    z = rng.standard_normal((b, L, D))
    Dk = rng.standard_normal(D)
    A = -rng.uniform(0.5, 8, (D, N))
    B = rng.standard_normal((b, L, N))
    C = rng.standard_normal((b, L, N))
    h0 = rng.standard_normal((b, D, N))
    y, last = o.selective_scan_fwd(u, np.zeros((b, L, D)), A, B, C, D=Dk, z=z, delta_softplus=False, h0=h0)
    assert np.array_equal(last, h0)
    ref = np.einsum("bln,bdn->bld", C, h0) + Dk * u
    assert _rel(y, ref * _silu(z)) < 1e-13
    y0, last0 = o.selective_scan_fwd(u, np.zeros((b, L, D)), A, B, C, D=Dk, z=z, delta_softplus=False)
    assert np.all(last0 == 0.0)
    assert _rel(y0, Dk * u * _silu(z)) < 1e-14
    ys, st = o.state_update(h0, u[:, 0], np.zeros((b, D)), A, B[:, 0], C[:, 0], D=Dk, z=z[:, 0])
    assert np.array_equal(st, h0)


def pin_scalar_closed_form(o):
    """Constant input to a single active state: h_t = b (1 - a^t) / (1 - a), the
    geometric sum of the recurrence h_t = a h_{t-1} + b ("Arch 02: Mamba SSM")."""
    L, D, N = 50, 3, 4
    A = -np.array([[0.7, 2, 3, 4], [1.3, 2, 3, 4], [0.05, 1, 1, 1]])
    dts = np.array([0.3, 0.11, 0.9])
    u0, B0, C0 = 1.7, -0.6, 1.9
    Dk = np.array([0.5, -1.0, 2.0])
    Bm = np.zeros((1, L, N))
    Bm[..., 0] = B0
    Cm = np.full((1, L, N), 5.0)  # C on the inactive states multiplies zeros
    Cm[..., 0] = C0
    y, last = o.selective_scan_fwd(np.full((1, L, D), u0), np.broadcast_to(dts, (1, L, D)), A, Bm, Cm,
                                   D=Dk, delta_softplus=False)
    t = np.arange(1, L + 1)[:, None]
    a = np.exp(dts * A[:, 0])
    bb = dts * B0 * u0
    h = bb * (1 - a ** t) / (1 - a)
    assert _rel(y[0], C0 * h + Dk * u0) < 1e-12
    assert _rel(last[0, :, 0], h[-1]) < 1e-12
    assert np.all(last[0, :, 1:] == 0.0)


def pin_bruteforce_unrolling(o, seed=3):
    """Tiny L: h_t = sum_{s<=t} (prod_{r=s+1..t} A-bar_r) B-bar_s u_s with explicit
    products ("Arch 02: Mamba SSM" recurrence; "8.7 State Space Models (Mamba)" 2.1)."""
    rng = np.random.default_rng(seed)
    b, L, D, N = 2, 6, 3, 4
    u = rng.standard_normal((b, L, D))
    raw = rng.normal(-1, 1, (b, L, D))
    bias = rng.normal(0, 0.5, D)
    z = rng.standard_normal((b, L, D))
    A = -rng.uniform(0.1, 4, (D, N))
    B = rng.standard_normal((b, L, N))
    C = rng.standard_normal((b, L, N))
    Dk = rng.standard_normal(D)
    y, last = o.selective_scan_fwd(u, raw, A, B, C, D=Dk, z=z, delta_bias=bias, delta_softplus=True)
    ref = np.zeros((b, L, D))
    hL = np.zeros((b, D, N))
    for bi in range(b):
        for d in range(D):
            dt = _softplus(raw[bi, :, d] + bias[d])
            for t in range(L):
                h = np.zeros(N)
                for s in range(t + 1):
                    prod = np.ones(N)
                    for r in range(s + 1, t + 1):
                        prod = prod * np.exp(dt[r] * A[d])
                    h += prod * dt[s] * B[bi, s] * u[bi, s, d]
                ref[bi, t, d] = (np.dot(C[bi, t], h) + Dk[d] * u[bi, t, d]) * _silu(z[bi, t, d])
                if t == L - 1:
                    hL[bi, d] = h
    assert _rel(y, ref) < 1e-12, _rel(y, ref)
    assert _rel(last, hL) < 1e-12


def pin_large_delta_reset(o, seed=4):
    """Large Delta replaces the state by the current write ("Arch 02: Mamba SSM": large
    Delta ~ full state replacement; "Mamba and State Space Models", worked pass)."""
    rng = np.random.default_rng(seed)
    b, L, D, N = 1, 7, 3, 4
    u = rng.standard_normal((b, L, D))
    A = -rng.uniform(1, 3, (D, N))
    B = rng.standard_normal((b, L, N))
    C = rng.standard_normal((b, L, N))
    big = 50.0
    y, last = o.selective_scan_fwd(u, np.full((b, L, D), big), A, B, C, delta_softplus=False)
    h = big * B[:, :, None, :] * u[:, :, :, None]  # (b, L, D, N)
    ref = np.einsum("bln,bldn->bld", C, h)
    assert _rel(y, ref) < 1e-15 + 1e-20
    assert _rel(last, h[:, -1]) < 1e-15


def pin_stability_bound(o, seed=5):
    """Delta > 0 and A < 0 give 0 < A-bar < 1 and a bounded state:
    |h_t[n]| <= max|B-bar u| / (1 - max A-bar) ("Mamba and State Space Models",
    "Discretization and initialization details": exp(Delta A) in (0,1), stable)."""
    rng = np.random.default_rng(seed)
    b, L, D, N = 1, 40, 3, 4
    u = rng.standard_normal((b, L, D)) * 3
    raw = rng.normal(-1, 1, (b, L, D))
    A = -rng.uniform(0.3, 2, (D, N))
    B = rng.standard_normal((b, L, N))
    C = rng.standard_normal((b, L, N))
    dt = _softplus(raw)
    abar = np.exp(dt[..., None] * A[None, None])           # (b, L, D, N)
    assert np.all((abar > 0) & (abar < 1))
    bmax = np.max(np.abs(dt[..., None] * B[:, :, None, :] * u[..., None]), axis=1)  # (b, D, N)
    bound = bmax / (1 - np.max(abar, axis=1))
    for Lp in range(1, L + 1):
        _, last = o.selective_scan_fwd(u[:, :Lp], raw[:, :Lp], A, B[:, :Lp], C[:, :Lp], delta_softplus=True)
        assert np.all(np.abs(last) <= bound * (1 + 1e-12))


def pin_decode_matches_forward(o, seed=6):
    """T single-token updates from zero == forward over T steps; and the state after a
    prefix continues the sequence ("Mamba and State Space Models", "Common Pitfalls":
    the state after a shared prefix is reusable; "8.7 State Space Models (Mamba)" s.5)."""
    rng = np.random.default_rng(seed)
    b, L, D, N = 2, 12, 3, 8
    u = rng.standard_normal((b, L, D))
    dt = _softplus(rng.standard_normal((b, L, D)))
    z = rng.standard_normal((b, L, D))
    A = -rng.uniform(0.1, 4, (D, N))
    B = rng.standard_normal((b, L, N))
    C = rng.standard_normal((b, L, N))
    Dk = rng.standard_normal(D)
    y, last = o.selective_scan_fwd(u, dt, A, B, C, D=Dk, z=z, delta_softplus=False)
    st = np.zeros((b, D, N))
    for t in range(L):
        yt, st = o.state_update(st, u[:, t], dt[:, t], A, B[:, t], C[:, t], D=Dk, z=z[:, t])
        assert _rel(yt, y[:, t]) < 1e-14
    assert _rel(st, last) < 1e-14
    P = 5
    _, mid = o.selective_scan_fwd(u[:, :P], dt[:, :P], A, B[:, :P], C[:, :P], D=Dk, z=z[:, :P],
                                  delta_softplus=False)
    y2, last2 = o.selective_scan_fwd(u[:, P:], dt[:, P:], A, B[:, P:], C[:, P:], D=Dk, z=z[:, P:],
                                     delta_softplus=False, h0=mid)
    assert _rel(y2, y[:, P:]) < 1e-14 and _rel(last2, last) < 1e-14


def pin_softplus_silu(o):
    """Softplus = log(1 + e^r) and SiLU = z sigmoid(z), against library routines and
    exact values (softplus(0) = ln 2; silu(0) = 0)."""
    assert abs(o.softplus(0.0) - np.log(2.0)) < 1e-16
    for r in np.linspace(-60, 60, 241):
        ref = _softplus(r)
        assert abs(o.softplus(r) - ref) <= 1e-15 * max(abs(ref), 1e-300), r
    assert o.silu(0.0) == 0.0
    for zz in np.linspace(-40, 40, 161):
        ref = _silu(zz)
        assert abs(o.silu(zz) - ref) <= 1e-15 * max(abs(ref), 1e-300) + 1e-300, zz


def combine(p, q):
    """The scan operator on (a, b) pairs: applying (a1, b1) then (a2, b2) to a state h
    gives a2 (a1 h + b1) + b2 = (a1 a2) h + (a2 b1 + b2)."""
    return p[0] * q[0], q[0] * p[1] + q[1]


def pin_scan_operator(o, seed=7):
    """The recurrence h_t = a_t h_{t-1} + b_t is a fold of an associative operator
    ("8.7 State Space Models (Mamba)", section 4.1; "Mamba and State Space Models",
    "Hardware-Aware Parallel Scan"), and the fold reproduces the oracle's state."""
    rng = np.random.default_rng(seed)
    for _ in range(200):
        p, q, r = [(rng.uniform(0, 1), rng.standard_normal()) for _ in range(3)]
        lhs = combine(combine(p, q), r)
        rhs = combine(p, combine(q, r))
        assert abs(lhs[0] - rhs[0]) <= 1e-15 and abs(lhs[1] - rhs[1]) <= 1e-14 * (1 + abs(lhs[1]))
    L, N = 33, 4
    u = rng.standard_normal((1, L, 1))
    dt = _softplus(rng.standard_normal((1, L, 1)))
    A = -rng.uniform(0.1, 2, (1, N))
    B = rng.standard_normal((1, L, N))
    C = rng.standard_normal((1, L, N))
    _, last = o.selective_scan_fwd(u, dt, A, B, C, delta_softplus=False)
    acc = (np.ones(N), np.zeros(N))
    for t in range(L):
        acc = combine(acc, (np.exp(dt[0, t, 0] * A[0]), dt[0, t, 0] * B[0, t] * u[0, t, 0]))
    assert _rel(last[0, 0], acc[1]) < 1e-13


def pin_decode_step_map(o, seed=8):
    """The decode step with the forward pass's step-size map (dt = softplus(delta + bias),
    "Mamba and State Space Models", "Discretization and initialization details") equals
    the plain step given dt computed here with numpy, and equals one forward step from
    the same start state with the same bias and softplus."""
    rng = np.random.default_rng(seed)
    b, D, N = 3, 5, 8
    st0 = rng.standard_normal((b, D, N))
    x = rng.standard_normal((b, D))
    raw = rng.standard_normal((b, D)) * 2
    bias = rng.uniform(-3, 1, D)
    z = rng.standard_normal((b, D))
    A = -rng.uniform(0.1, 4, (D, N))
    B = rng.standard_normal((b, N))
    C = rng.standard_normal((b, N))
    Dk = rng.standard_normal(D)
    ye, se = o.state_update(st0, x, raw, A, B, C, D=Dk, z=z, delta_bias=bias, delta_softplus=True)
    yp, sp = o.state_update(st0, x, _softplus(raw + bias), A, B, C, D=Dk, z=z)
    assert _rel(ye, yp) < 1e-14 and _rel(se, sp) < 1e-14
    yf, sf = o.selective_scan_fwd(x[:, None], raw[:, None], A, B[:, None], C[:, None], D=Dk, z=z[:, None],
                                  delta_bias=bias, delta_softplus=True, h0=st0)
    assert _rel(ye, yf[:, 0]) < 1e-14 and _rel(se, sf) < 1e-14
    # bias without softplus: dt = delta + bias exactly
    yb, sb = o.state_update(st0, x, raw, A, B, C, D=Dk, z=z, delta_bias=bias, delta_softplus=False)
    yq, sq = o.state_update(st0, x, raw + bias, A, B, C, D=Dk, z=z)
    assert _rel(yb, yq) < 1e-15 and _rel(sb, sq) < 1e-15


def pin_zoh_solves_the_ode(o, seed=9):
    """With zoh, each step is the exact solution of the continuous system
    dh/ds = A h + B_t u_t over a step of length dt_t with the input held constant
    ("Arch 02: Mamba SSM", zero-order hold; "8.7 State Space Models (Mamba)", section 3).
    Checked against a numerical ODE integration of that system."""
    from scipy.integrate import solve_ivp
    rng = np.random.default_rng(seed)
    L, D, N = 6, 2, 4
    u = rng.standard_normal((1, L, D))
    dt = rng.uniform(0.05, 0.8, (1, L, D))
    A = -rng.uniform(0.2, 3.0, (D, N))
    B = rng.standard_normal((1, L, N))
    C = rng.standard_normal((1, L, N))
    y, last = o.selective_scan_fwd(u, dt, A, B, C, delta_softplus=False, zoh=True)
    for d in range(D):
        h = np.zeros(N)
        for t in range(L):
            f = lambda s, hh, t=t, d=d: A[d] * hh + B[0, t] * u[0, t, d]
            h = solve_ivp(f, (0.0, dt[0, t, d]), h, method="DOP853", rtol=1e-12, atol=1e-14).y[:, -1]
            assert abs(y[0, t, d] - C[0, t] @ h) <= 1e-9 * (1 + abs(y[0, t, d]))
        assert np.max(np.abs(last[0, d] - h)) <= 1e-9 * (1 + np.max(np.abs(h)))


def pin_zoh_limits(o, seed=10):
    """The zero-order-hold B-bar (exp(dt a) - 1) / a B tends to dt B as dt a -> 0 (the
    simplification the pages take for Mamba) and equals it where a = 0."""
    rng = np.random.default_rng(seed)
    b, L, D, N = 1, 9, 3, 4
    u = rng.standard_normal((b, L, D))
    B = rng.standard_normal((b, L, N))
    C = rng.standard_normal((b, L, N))
    A = -rng.uniform(0.5, 2.0, (D, N))
    A[1, 2] = 0.0
    dt = rng.uniform(0.5, 1.0, (b, L, D))
    yz, lz = o.selective_scan_fwd(u, dt, A, B, C, delta_softplus=False, zoh=True)
    yd, ld = o.selective_scan_fwd(u, dt, A, B, C, delta_softplus=False)
    assert _rel(lz, ld) > 1e-2  # the two discretisations differ at finite dt
    A0 = np.zeros_like(A)
    y0z, l0z = o.selective_scan_fwd(u, dt, A0, B, C, delta_softplus=False, zoh=True)
    y0d, l0d = o.selective_scan_fwd(u, dt, A0, B, C, delta_softplus=False)
    assert _rel(y0z, y0d) < 1e-15 and _rel(l0z, l0d) < 1e-15
    eps = 1e-7
    ys, ls = o.selective_scan_fwd(u, dt * eps, A, B, C, delta_softplus=False, zoh=True)
    ysd, lsd = o.selective_scan_fwd(u, dt * eps, A, B, C, delta_softplus=False)
    assert _rel(ls, lsd) < 1e-6
    # decode with zoh == one forward step with zoh
    st0 = rng.standard_normal((b, D, N))
    ye, se = o.state_update(st0, u[:, 0], dt[:, 0], A, B[:, 0], C[:, 0], zoh=True)
    yf, sf = o.selective_scan_fwd(u[:, :1], dt[:, :1], A, B[:, :1], C[:, :1], delta_softplus=False, zoh=True, h0=st0)
    assert _rel(ye, yf[:, 0]) < 1e-14 and _rel(se, sf) < 1e-14


def pin_conv_prologue(o, seed=11):
    """The causal depthwise width-4 convolution + SiLU before the SSM ("Mamba and State
    Space Models", "The Mamba Block") against numpy's convolution: u_t uses x_{t-3..t},
    with the carried conv state (the three inputs before the sequence) or zeros in front;
    and a sequence cut anywhere continues exactly from the next conv state."""
    rng = np.random.default_rng(seed)
    b, L, D = 2, 11, 3
    x = rng.standard_normal((b, L, D))
    w = rng.standard_normal((D, 4))
    bias = rng.standard_normal(D)
    cs = rng.standard_normal((b, D, 3))
    for state in (None, cs):
        u = o.conv1d_silu(x, w, bias, state)
        for bi in range(b):
            for d in range(D):
                front = np.zeros(3) if state is None else state[bi, d]
                seq = np.concatenate([front, x[bi, :, d]])
                ref = np.convolve(seq, w[d][::-1])[3:3 + L] + bias[d]
                assert np.max(np.abs(u[bi, :, d] - _silu(ref))) <= 1e-14 * (1 + np.max(np.abs(ref)))
    u_all = o.conv1d_silu(x, w, bias, cs)
    for P in (1, 2, 5):
        nxt = o.next_conv_state(x[:, :P], cs)
        u_rest = o.conv1d_silu(x[:, P:], w, bias, nxt)
        assert np.array_equal(u_rest, u_all[:, P:])
    assert np.array_equal(o.next_conv_state(x, cs), np.transpose(x[:, -3:], (0, 2, 1)))
    A = -rng.uniform(0.5, 2.0, (D, 4))
    Bm = rng.standard_normal((b, L, 4))
    Cm = rng.standard_normal((b, L, 4))
    dt = rng.uniform(0.01, 0.5, (b, L, D))
    y, last, nxt = o.conv_selective_scan_fwd(x, w, A, Bm, Cm, dt, conv_bias=bias, conv_state=cs,
                                             delta_softplus=False)
    y2, last2 = o.selective_scan_fwd(u_all, dt, A, Bm, Cm, delta_softplus=False)
    assert np.array_equal(y, y2) and np.array_equal(last, last2)


def pin_backward_finite_differences(o, seed=12):
    """The backward pass against central finite differences of the forward pass: for the
    loss sum(dy * y) + sum(dlast * last_state), every element of every input."""
    rng = np.random.default_rng(seed)
    b, L, D, N = 2, 7, 3, 4
    base = dict(u=rng.standard_normal((b, L, D)), delta=rng.standard_normal((b, L, D)) * 0.5 - 1.0,
                A=-rng.uniform(0.3, 2.0, (D, N)), B=rng.standard_normal((b, L, N)), C=rng.standard_normal((b, L, N)),
                D=rng.standard_normal(D), z=rng.standard_normal((b, L, D)), delta_bias=rng.uniform(-0.5, 0.5, D),
                h0=rng.standard_normal((b, D, N)))
    dy = rng.standard_normal((b, L, D))
    dlast = rng.standard_normal((b, D, N))
    for softplus, keys in ((True, list(base)), (False, ["u", "delta", "A", "B", "C"])):
        inp = {k: base[k] for k in keys}
        if not softplus:
            inp["delta"] = np.abs(base["delta"]) + 0.05  # a positive step size

        def loss(x):
            y, last = o.selective_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x.get("D"), z=x.get("z"),
                                           delta_bias=x.get("delta_bias"), delta_softplus=softplus, h0=x.get("h0"))
            return float(np.sum(dy * y) + np.sum(dlast * last))

        gr = o.selective_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dy, D=inp.get("D"),
                                  z=inp.get("z"), delta_bias=inp.get("delta_bias"), delta_softplus=softplus,
                                  h0=inp.get("h0"), dlast=dlast)
        names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "z": "dz",
                 "delta_bias": "dbias", "h0": "dh0"}
        eps = 1e-6
        for k in keys:
            g = gr[names[k]]
            for idx in np.ndindex(inp[k].shape):
                xp = {kk: v.copy() for kk, v in inp.items()}
                xm = {kk: v.copy() for kk, v in inp.items()}
                xp[k][idx] += eps
                xm[k][idx] -= eps
                fd = (loss(xp) - loss(xm)) / (2 * eps)
                assert abs(fd - g[idx]) <= 1e-6 * (1 + abs(fd)), (k, idx, fd, g[idx])


def pin_ssd_duality_and_mamba1(o, seed=13):
    """Mamba-2 SSD ("Mamba and State Space Models", "Mamba-2 and State Space Duality"):
    (1) the recurrence equals the masked quadratic form Y = tril(C B^T o M) (dt X) + D X
    with M_ji = prod_{k=i+1..j} a_k, computed here by brute force with explicit products;
    (2) with P = 1 every (head, p) is a Mamba-1 channel whose N states share the head's A,
    so the result equals the (separately pinned) Mamba-1 oracle on those channels."""
    rng = np.random.default_rng(seed)
    b, L, H, P, N, G = 2, 9, 4, 3, 5, 2
    x = rng.standard_normal((b, L, H, P))
    raw = rng.standard_normal((b, L, H)) * 0.5
    A = -rng.uniform(0.2, 2.0, H)
    B = rng.standard_normal((b, L, G, N))
    C = rng.standard_normal((b, L, G, N))
    Dk = rng.standard_normal(H)
    bias = rng.uniform(-0.5, 0.5, H)
    h0 = rng.standard_normal((b, H, P, N))
    y, last = o.ssd_fwd(x, raw, A, B, C, D=Dk, dt_bias=bias, dt_softplus=True, h0=h0)
    dt = _softplus(raw + bias)
    for bi in range(b):
        for h in range(H):
            g = h // (H // G)
            a = np.exp(dt[bi, :, h] * A[h])
            Yr = np.zeros((L, P))
            for j in range(L):
                pre = np.prod(a[:j + 1])                      # decay of h0 up to step j
                Yr[j] += (h0[bi, h] @ C[bi, j, g]) * pre
                for i in range(j + 1):
                    m = np.prod(a[i + 1:j + 1])               # M_ji
                    Yr[j] += (C[bi, j, g] @ B[bi, i, g]) * m * dt[bi, i, h] * x[bi, i, h]
                Yr[j] += Dk[h] * x[bi, j, h]
            assert _rel(y[bi, :, h], Yr) < 1e-13
    # P = 1: Mamba-1 channels with a per-head A repeated over the N states
    x1 = x[..., :1]
    y1, l1 = o.ssd_fwd(x1, raw, A, B, C, D=Dk, dt_bias=bias, dt_softplus=True)
    for g in range(G):
        hs = list(range(g * (H // G), (g + 1) * (H // G)))
        ym, lm = o.selective_scan_fwd(x1[:, :, hs, 0], raw[:, :, hs], np.repeat(A[hs, None], N, axis=1),
                                      B[:, :, g], C[:, :, g], D=Dk[hs], delta_bias=bias[hs], delta_softplus=True)
        assert _rel(y1[:, :, hs, 0], ym) < 1e-13 and _rel(l1[:, hs, 0, :], lm) < 1e-13


ALL_PINS = [pin_worked_example, pin_lti_convolution, pin_delta_zero_holds_state, pin_scalar_closed_form,
            pin_bruteforce_unrolling, pin_large_delta_reset, pin_stability_bound, pin_decode_matches_forward,
            pin_softplus_silu, pin_scan_operator, pin_decode_step_map, pin_zoh_solves_the_ode, pin_zoh_limits,
            pin_conv_prologue, pin_backward_finite_differences, pin_ssd_duality_and_mamba1]
