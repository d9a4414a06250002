"""Independent checks that pin the oracle to mathematics it does not itself use.

Each ``check_*`` function returns the worst error it found (a float); the
tests compare it with a bound.  None of them re-types the oracle's recursion:
they use a closed-form (non-recursive) sum, finite differences, textbook
special cases (geometric series, causal convolution), limits, invariants and
a hand-worked example.  The mutation test reuses them to show that a planted
mistake in a copy of the oracle source fails at least one.
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit

import oracle


# --------------------------------------------------------------- inputs

def rand_problem(B, L, D, N, seed, *, with_z=True, with_h0=True, with_dh_last=True,
                 bias_scale=1.0):
    """Random f64 problem with O(1) Δ so that the decay is neither ~0 nor ~1."""
    r = np.random.default_rng(seed)
    p = {
        "u": r.standard_normal((B, L, D)),
        "delta_raw": r.standard_normal((B, L, D)),
        "z": r.standard_normal((B, L, D)) if with_z else None,
        "Bm": r.standard_normal((B, L, N)),
        "Cm": r.standard_normal((B, L, N)),
        "A_log": 0.5 * r.standard_normal((D, N)),
        "Dp": r.standard_normal(D),
        "delta_bias": bias_scale * r.standard_normal(D),
        "h0": r.standard_normal((B, D, N)) if with_h0 else None,
    }
    dout = r.standard_normal((B, L, D))
    dh_last = r.standard_normal((B, D, N)) if with_dh_last else None
    return p, dout, dh_last


def _fwd(p, dt_limit=None):
    return oracle.fwd(p["u"], p["delta_raw"], p["z"], p["Bm"], p["Cm"], p["A_log"], p["Dp"],
                      p["delta_bias"], p["h0"], threads=1, dt_limit=dt_limit)


def _bwd(p, dout, dh_last, dt_limit=None):
    return oracle.bwd(p["u"], p["delta_raw"], p["z"], p["Bm"], p["Cm"], p["A_log"], p["Dp"],
                      p["delta_bias"], p["h0"], dout, dh_last, threads=1, dt_limit=dt_limit)


# --------------------------------------------------------------- closed form

def closed_form_forward(p):
    """Non-recursive S6 forward:  h_t = e^{A S_t} h0 + sum_{k<=t} e^{A (S_t - S_k)} Δ_k B_k u_k,
    S_t = sum_{j<=t} Δ_j, with softplus written as logaddexp(0, s) and the gate via expit."""
    u, B_, C_ = p["u"], p["Bm"], p["Cm"]
    Bsz, L, D = u.shape
    N = B_.shape[2]
    A = -np.exp(p["A_log"])                                   # [D, N]
    delta = np.logaddexp(0.0, p["delta_raw"] + p["delta_bias"][None, None, :])  # [B, L, D]
    S = np.cumsum(delta, axis=1)                              # [B, L, D]
    h0 = p["h0"] if p["h0"] is not None else np.zeros((Bsz, D, N))
    out = np.empty((Bsz, L, D))
    h_last = np.empty((Bsz, D, N))
    for b in range(Bsz):
        for t in range(L):
            # decay[k, d, n] = exp(A[d,n] * (S_t - S_k)) for k <= t
            dec = np.exp(A[None, :, :] * (S[b, t, :][None, :, None] - S[b, : t + 1, :][:, :, None]))
            src = (delta[b, : t + 1, :] * u[b, : t + 1, :])[:, :, None] * B_[b, : t + 1, None, :]
            h = np.exp(A * S[b, t, :][:, None]) * h0[b] + (dec * src).sum(axis=0)  # [D, N]
            y = (h * C_[b, t, None, :]).sum(axis=1) + p["Dp"] * u[b, t]
            out[b, t] = y if p["z"] is None else y * p["z"][b, t] * expit(p["z"][b, t])
            if t == L - 1:
                h_last[b] = h
    return out, h_last


def check_closed_form(seed=0, shape=(2, 9, 3, 5), **kw):
    p, _, _ = rand_problem(*shape, seed, **kw)
    out, h_last = _fwd(p)
    ref_out, ref_h = closed_form_forward(p)
    e1 = np.max(np.abs(out - ref_out)) / np.max(np.abs(ref_out))
    e2 = np.max(np.abs(h_last - ref_h)) / np.max(np.abs(ref_h))
    return max(e1, e2)


# --------------------------------------------------------------- finite differences

def _loss(p, dout, dh_last, dt_limit=None):
    out, h_last = _fwd(p, dt_limit)
    v = float(np.sum(dout * out))
    if dh_last is not None:
        v += float(np.sum(dh_last * h_last))
    return v


GRAD_OF = {"u": "du", "delta_raw": "d_delta_raw", "z": "dz", "Bm": "dBm", "Cm": "dCm",
           "A_log": "dA_log", "Dp": "dD", "delta_bias": "d_delta_bias", "h0": "dh0"}


def check_finite_differences(seed=0, shape=(2, 7, 3, 2), eps=1e-6, dt_limit=None, p=None, **kw):
    """max over inputs of  max|fd - analytic| / max|analytic|  (central differences)."""
    if p is None:
        p, dout, dh_last = rand_problem(*shape, seed, **kw)
    else:
        p, dout, dh_last = p
    g = _bwd(p, dout, dh_last, dt_limit)
    worst = 0.0
    for name, gname in GRAD_OF.items():
        x = p[name]
        if x is None:
            continue
        fd = np.empty_like(x)
        flat = x.reshape(-1)
        fdf = fd.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            h = eps * max(1.0, abs(old))
            flat[i] = old + h
            lp = _loss(p, dout, dh_last, dt_limit)
            flat[i] = old - h
            lm = _loss(p, dout, dh_last, dt_limit)
            flat[i] = old
            fdf[i] = (lp - lm) / (2 * h)
        an = g[gname]
        scale = max(np.max(np.abs(fd)), 1e-30)
        worst = max(worst, float(np.max(np.abs(fd - an)) / scale))
    return worst


# --------------------------------------------------------------- special cases

def check_geometric_series(L=40, N=3):
    """Constant u, Δ, B, C, z: h_t = ΔBu (1 - a^{t+1}) / (1 - a), a = e^{ΔA}."""
    D = 2
    u0, raw0, B0, C0, z0 = 0.7, 0.3, np.array([1.5, -0.4, 0.9]), np.array([0.2, 1.1, -0.6]), 0.8
    A_log = np.tile(np.log(np.arange(1, N + 1, dtype=float)), (D, 1))
    p = {"u": np.full((1, L, D), u0), "delta_raw": np.full((1, L, D), raw0),
         "z": np.full((1, L, D), z0), "Bm": np.tile(B0[:N], (1, L, 1)),
         "Cm": np.tile(C0[:N], (1, L, 1)), "A_log": A_log, "Dp": np.array([0.5, -1.0]),
         "delta_bias": np.zeros(D), "h0": None}
    out, h_last = _fwd(p)
    delta = np.log1p(np.exp(raw0))
    a = np.exp(-delta * np.arange(1, N + 1))
    t = np.arange(L)[:, None]
    h = delta * B0[:N] * u0 * (1 - a[None, :] ** (t + 1)) / (1 - a[None, :])  # [L, N]
    y = h @ C0[:N]                                                           # [L]
    gate = z0 * expit(z0)
    ref = (y[:, None] + p["Dp"][None, :] * u0) * gate                         # [L, D]
    lim = delta * B0[:N] * u0 / (1 - a)
    e1 = np.max(np.abs(out[0] - ref)) / np.max(np.abs(ref))
    e2 = np.max(np.abs(h_last[0] - lim[None, :])) / np.max(np.abs(lim))  # L=40: a^41 ~ 0
    return max(e1, e2 if L >= 40 else 0.0)


def check_delta_zero(seed=3):
    """delta_raw = -800 makes softplus underflow to exactly 0: y = Dp*u, h_last = h0."""
    p, _, _ = rand_problem(2, 6, 3, 4, seed)
    p["delta_raw"][:] = -800.0
    p["delta_bias"][:] = 0.0
    out, h_last = _fwd(p)
    y = p["Dp"][None, None, :] * p["u"] + np.einsum("bdn,bln->bld", p["h0"], p["Cm"])
    ref = y * p["z"] * expit(p["z"])
    return max(float(np.max(np.abs(out - ref))), float(np.max(np.abs(h_last - p["h0"]))))


def check_state_reset(seed=4):
    """A_log = 60 gives a = exp(-Δ e^60) = 0: the state forgets, h_t = Δ_t B_t u_t."""
    p, _, _ = rand_problem(2, 6, 3, 4, seed)
    p["A_log"][:] = 60.0
    out, h_last = _fwd(p)
    delta = np.logaddexp(0.0, p["delta_raw"] + p["delta_bias"])
    y = np.einsum("bln,bln->bl", p["Bm"], p["Cm"])[:, :, None] * delta * p["u"] + p["Dp"] * p["u"]
    ref = y * p["z"] * expit(p["z"])
    h_ref = (delta[:, -1, :] * p["u"][:, -1, :])[:, :, None] * p["Bm"][:, -1, None, :]
    return max(float(np.max(np.abs(out - ref)) / np.max(np.abs(ref))),
               float(np.max(np.abs(h_last - h_ref)) / np.max(np.abs(h_ref))))


def check_lti_convolution(L=50, seed=5):
    """Δ, B, C constant in time: y = causal convolution of u with K_k = Σ_n C Δ B a_n^k."""
    r = np.random.default_rng(seed)
    N, D = 4, 2
    u = r.standard_normal((1, L, D))
    B0, C0 = r.standard_normal(N), r.standard_normal(N)
    A_log = 0.3 * r.standard_normal((D, N))
    raw0 = np.array([0.2, -0.5])
    p = {"u": u, "delta_raw": np.tile(raw0, (1, L, 1)), "z": None, "Bm": np.tile(B0, (1, L, 1)),
         "Cm": np.tile(C0, (1, L, 1)), "A_log": A_log, "Dp": np.array([0.3, 1.7]),
         "delta_bias": np.zeros(D), "h0": None}
    out, _ = _fwd(p)
    worst = 0.0
    for d in range(D):
        delta = np.log1p(np.exp(raw0[d]))
        a = np.exp(-np.exp(A_log[d]) * delta)
        K = np.array([np.sum(C0 * delta * B0 * a ** k) for k in range(L)])
        ref = np.convolve(u[0, :, d], K)[:L] + p["Dp"][d] * u[0, :, d]
        worst = max(worst, float(np.max(np.abs(out[0, :, d] - ref)) / np.max(np.abs(ref))))
    return worst


def check_hand_worked(fixture):
    """The hand-derived example stored under tests/golden/ (see its derivation)."""
    inp = fixture["inputs"]
    p = {k: (np.array(v, dtype=float) if v is not None else None) for k, v in inp.items()}
    out, h_last = _fwd(p)
    e = np.max(np.abs(out.reshape(-1) - np.array(fixture["expected"]["out"]).reshape(-1)))
    e2 = np.max(np.abs(h_last.reshape(-1) - np.array(fixture["expected"]["h_last"]).reshape(-1)))
    return float(max(e, e2))


def check_internal_consistency(seed=6):
    """d_delta_bias = Σ_{b,t} d_delta_raw and dD = Σ_{b,t} dy*u with dy = dout*silu(z)."""
    p, dout, dh_last = rand_problem(3, 8, 4, 3, seed)
    g = _bwd(p, dout, dh_last)
    dy = dout * p["z"] * expit(p["z"])
    e1 = np.max(np.abs(g["d_delta_bias"] - g["d_delta_raw"].sum(axis=(0, 1))))
    e2 = np.max(np.abs(g["dD"] - (dy * p["u"]).sum(axis=(0, 1))))
    return float(max(e1, e2))


# --------------------------------------------------------------- the limit on Δ

def _softplus(s):
    return np.logaddexp(0.0, s)


def dt_limit_problem(B, L, D, N, seed, lo_q=0.3, hi_q=0.7, margin=1e-3):
    """A random problem and a limit [dt_min, dt_max] at the lo_q / hi_q
    quantiles of its Δ = softplus(s), so that both ends clamp; every s whose
    softplus lies within ``margin`` of a limit is moved off it (a finite
    difference or an f32 rounding must not cross a kink)."""
    p, dout, dh_last = rand_problem(B, L, D, N, seed)
    sp = _softplus(p["delta_raw"] + p["delta_bias"])
    lo, hi = np.quantile(sp, lo_q), np.quantile(sp, hi_q)
    for _ in range(8):
        sp = _softplus(p["delta_raw"] + p["delta_bias"])
        near = (np.abs(sp - lo) < margin) | (np.abs(sp - hi) < margin)
        if not near.any():
            break
        p["delta_raw"][near] += 4 * margin
    return (p, dout, dh_last), (float(lo), float(hi))


def check_dt_limit_finite_differences(seed=11):
    """With both ends of the limit active: every gradient against central
    differences of the clamped loss (the clamped steps give delta_raw and
    delta_bias no gradient; du, dB, dA_log use the clamped Δ)."""
    prob, lim = dt_limit_problem(2, 7, 3, 2, seed)
    return check_finite_differences(p=prob, dt_limit=lim)


def check_dt_limit_reparam(seed=12):
    """The limit acts on Δ = softplus(s): the clamped forward equals the
    unclamped forward of delta_raw' = softplus^-1(clamp(softplus(s))) - bias."""
    (p, _, _), (lo, hi) = dt_limit_problem(2, 9, 3, 4, seed, margin=0.0)
    out, h_last = _fwd(p, (lo, hi))
    s = p["delta_raw"] + p["delta_bias"]
    delta = np.clip(_softplus(s), lo, hi)
    q = dict(p)
    q["delta_raw"] = np.log(np.expm1(delta)) - p["delta_bias"]
    ref_out, ref_h = _fwd(q)
    return max(float(np.max(np.abs(out - ref_out)) / np.max(np.abs(ref_out))),
               float(np.max(np.abs(h_last - ref_h)) / np.max(np.abs(ref_h))))


def check_dt_constant(L=40, N=3, seed=13):
    """dt_min = dt_max = c fixes Δ = c whatever delta_raw is: with constant
    u, B, C, z the state is the geometric series c B u (1 - a^{t+1}) / (1 - a),
    a = e^{c A}; and no gradient reaches delta_raw or delta_bias."""
    r = np.random.default_rng(seed)
    D, c = 2, 0.37
    u0, z0 = 0.7, 0.8
    B0, C0 = np.array([1.5, -0.4, 0.9])[:N], np.array([0.2, 1.1, -0.6])[:N]
    A_log = np.tile(np.log(np.arange(1, N + 1, dtype=float)), (D, 1))
    p = {"u": np.full((1, L, D), u0), "delta_raw": r.standard_normal((1, L, D)),
         "z": np.full((1, L, D), z0), "Bm": np.tile(B0, (1, L, 1)), "Cm": np.tile(C0, (1, L, 1)),
         "A_log": A_log, "Dp": np.array([0.5, -1.0]), "delta_bias": np.zeros(D), "h0": None}
    out, _ = _fwd(p, (c, c))
    a = np.exp(-c * np.arange(1, N + 1))
    t = np.arange(L)[:, None]
    h = c * B0 * u0 * (1 - a[None, :] ** (t + 1)) / (1 - a[None, :])
    ref = ((h @ C0)[:, None] + p["Dp"][None, :] * u0) * z0 * expit(z0)
    g = _bwd(p, r.standard_normal((1, L, D)), None, (c, c))
    return max(float(np.max(np.abs(out[0] - ref)) / np.max(np.abs(ref))),
               float(np.max(np.abs(g["d_delta_raw"]))), float(np.max(np.abs(g["d_delta_bias"]))))


ALL_CHECKS = {
    "closed_form": (lambda: check_closed_form(), 1e-12),
    "closed_form_nogate": (lambda: check_closed_form(seed=1, with_z=False, with_h0=False), 1e-12),
    "finite_differences": (lambda: check_finite_differences(), 1e-6),
    "finite_differences_nogate": (lambda: check_finite_differences(seed=2, with_z=False), 1e-6),
    "geometric_series": (lambda: check_geometric_series(), 1e-12),
    "delta_zero": (lambda: check_delta_zero(), 1e-14),
    "state_reset": (lambda: check_state_reset(), 1e-13),
    "lti_convolution": (lambda: check_lti_convolution(), 1e-12),
    "internal_consistency": (lambda: check_internal_consistency(), 1e-12),
    "dt_limit_finite_differences": (lambda: check_dt_limit_finite_differences(), 1e-6),
    "dt_limit_reparam": (lambda: check_dt_limit_reparam(), 1e-12),
    "dt_constant": (lambda: check_dt_constant(), 1e-12),
}
