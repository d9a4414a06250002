"""Pins for the Mamba-2 SSD oracle (CPU only): the reduction to the S6
oracle (head h, element p as S6 channel (h, p) with A[d][n] = A_h and the
group's B, C), the chunked matmul form written independently with numpy, a
closed form for constant inputs, delta fixed by dt_min = dt_max; for the
backward, central finite differences of every gradient (with and without a
limit on delta that clamps some steps), the reduction to the S6 oracle's
backward and the chunked matrix form of the backward written independently
in numpy; and planted mistakes that must each fail a pin."""
import os
import shutil

import numpy as np
import pytest

import oracle


def _problem(B=2, L=11, H=4, P=3, G=2, N=3, seed=0, h0=True):
    r = np.random.default_rng(seed)
    return {
        "x": r.standard_normal((B, L, H, P)),
        "dt_raw": r.standard_normal((B, L, H)),
        "dt_bias": 0.5 * r.standard_normal(H),
        "A_log": 0.4 * r.standard_normal(H),
        "Bm": r.standard_normal((B, L, G, N)),
        "Cm": r.standard_normal((B, L, G, N)),
        "Dp": r.standard_normal(H),
        "h0": r.standard_normal((B, H, N, P)) if h0 else None,
    }


def _ssd(p, dt_limit=None):
    return oracle.ssd_fwd(p["x"], p["dt_raw"], p["dt_bias"], p["A_log"], p["Bm"], p["Cm"], p["Dp"], p["h0"],
                          dt_limit=dt_limit)


def check_s6_reduction(dt_limit=None, seed=1):
    """Each group of heads is an S6 problem: channel d = (head, p) with
    u = x, delta_raw = dt_raw of the head, A_log[d][n] = A_log[head] for every
    n, the group's Bm / Cm, Dp[d] = Dp[head], h0[b][d][n] = h0[b][head][n][p]."""
    p = _problem(seed=seed)
    y, h_last = _ssd(p, dt_limit)
    B, L, H, P = p["x"].shape
    G, N = p["Bm"].shape[2], p["Bm"].shape[3]
    hpg = H // G
    err = 0.0
    for g in range(G):
        hs = slice(g * hpg, (g + 1) * hpg)
        u = p["x"][:, :, hs, :].reshape(B, L, hpg * P)
        raw = np.repeat(p["dt_raw"][:, :, hs], P, axis=2)
        bias = np.repeat(p["dt_bias"][hs], P)
        A_log = np.repeat(p["A_log"][hs], P)[:, None] * np.ones((1, N))
        Dp = np.repeat(p["Dp"][hs], P)
        h0 = np.transpose(p["h0"][:, hs], (0, 1, 3, 2)).reshape(B, hpg * P, N)
        out, hl = oracle.fwd(u, raw, None, p["Bm"][:, :, g, :], p["Cm"][:, :, g, :], A_log, Dp, bias, h0,
                             dt_limit=dt_limit)
        err = max(err, float(np.max(np.abs(out - y[:, :, hs, :].reshape(B, L, hpg * P)))))
        ref_h = np.transpose(hl.reshape(B, hpg, P, N), (0, 1, 3, 2))
        err = max(err, float(np.max(np.abs(ref_h - h_last[:, hs]))))
    return err


def chunked_form(p, Q):
    """The SSD's chunked matmul form (numpy): per chunk of Q steps, the
    intra-chunk term (C B^T masked by the decays between steps) times delta*x,
    plus the entering state read out through C with the decay to each step;
    chunk states handed on with the chunk's total decay."""
    x, Bm, Cm = p["x"], p["Bm"], p["Cm"]
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    hpg = H // G
    delta = np.logaddexp(0.0, p["dt_raw"] + p["dt_bias"])           # [B, L, H]
    A = -np.exp(p["A_log"])                                        # [H]
    y = np.empty_like(x)
    h_last = np.empty((B, H, N, P))
    for b in range(B):
        for h in range(H):
            g = h // hpg
            S = p["h0"][b, h].copy() if p["h0"] is not None else np.zeros((N, P))
            for c0 in range(0, L, Q):
                c1 = min(L, c0 + Q)
                dA = delta[b, c0:c1, h] * A[h]
                cum = np.cumsum(dA)                                   # log decay from chunk start
                Lmask = np.tril(np.exp(cum[:, None] - cum[None, :]))  # [t, s], s <= t
                CB = Cm[b, c0:c1, g] @ Bm[b, c0:c1, g].T              # [t, s]
                dx = delta[b, c0:c1, h][:, None] * x[b, c0:c1, h]     # [s, P]
                y_diag = (CB * Lmask) @ dx
                y_off = np.exp(cum)[:, None] * (Cm[b, c0:c1, g] @ S)
                y[b, c0:c1, h] = y_diag + y_off + p["Dp"][h] * x[b, c0:c1, h]
                w = np.exp(cum[-1] - cum)                             # decay from step s to chunk end
                S = np.exp(cum[-1]) * S + Bm[b, c0:c1, g].T @ (w[:, None] * dx)
            h_last[b, h] = S
    return y, h_last


def check_chunked_form(seed=2, Q=4):
    p = _problem(B=2, L=13, H=4, P=3, G=2, N=3, seed=seed)
    y, h_last = _ssd(p)
    ry, rh = chunked_form(p, Q)
    return max(float(np.max(np.abs(y - ry)) / np.max(np.abs(ry))),
               float(np.max(np.abs(h_last - rh)) / np.max(np.abs(rh))))


def _constant_problem(L, dt_raw=None):
    H, P, G, N = 2, 2, 1, 3
    x0 = np.array([[0.7, -0.3], [1.1, 0.4]])        # [H, P]
    B0 = np.array([1.5, -0.4, 0.9])
    C0 = np.array([0.2, 1.1, -0.6])
    p = {"x": np.tile(x0, (1, L, 1, 1)), "dt_raw": np.tile([0.3, -0.8], (1, L, 1)) if dt_raw is None else dt_raw,
         "dt_bias": np.zeros(H), "A_log": np.log(np.array([0.5, 2.0])),
         "Bm": np.tile(B0, (1, L, G, 1)), "Cm": np.tile(C0, (1, L, G, 1)), "Dp": np.array([0.5, -1.0]), "h0": None}
    return p, x0, B0, C0


def _geometric(delta, A, x0, B0, C0, Dp, L):
    """y_t = (C.B) delta x (1 - a^{t+1}) / (1 - a) + D x for constant inputs."""
    a = np.exp(delta * A)
    t = np.arange(L)
    return (C0 @ B0) * delta * x0 * ((1 - a ** (t + 1)) / (1 - a))[:, None] + Dp * x0


def check_closed_form(L=30):
    p, x0, B0, C0 = _constant_problem(L)
    y, _ = _ssd(p)
    err = 0.0
    for h in range(2):
        delta = np.log1p(np.exp(p["dt_raw"][0, 0, h]))
        ref = _geometric(delta, -np.exp(p["A_log"][h]), x0[h], B0, C0, p["Dp"][h], L)
        err = max(err, float(np.max(np.abs(y[0, :, h] - ref)) / np.max(np.abs(ref))))
    return err


def check_dt_fixed_by_limit(L=30, c=0.37):
    """dt_min = dt_max = c: delta = c whatever dt_raw is."""
    r = np.random.default_rng(9)
    p, x0, B0, C0 = _constant_problem(L, dt_raw=r.standard_normal((1, L, 2)))
    y, _ = _ssd(p, (c, c))
    err = 0.0
    for h in range(2):
        ref = _geometric(c, -np.exp(p["A_log"][h]), x0[h], B0, C0, p["Dp"][h], L)
        err = max(err, float(np.max(np.abs(y[0, :, h] - ref)) / np.max(np.abs(ref))))
    return err


_KEYS = ("x", "dt_raw", "dt_bias", "A_log", "Bm", "Cm", "Dp", "h0")
_GRAD = {"x": "dx", "dt_raw": "ddt_raw", "dt_bias": "ddt_bias", "A_log": "dA_log", "Bm": "dBm", "Cm": "dCm",
         "Dp": "dDp", "h0": "dh0"}


def chunked_backward(p, dy, dhl, Q):
    """The backward in the chunked matrix form (numpy), per chunk of Q steps
    walked last to first with dS = the gradient of the state leaving the
    chunk: with L the masked decays, CB = C B^T, Z[t][s] = dy_t . x_s,
    w_s = e^(cum_end - cum_s) and dec = e^(cum_end),
      dx = D dy + diag(delta) (L o CB)^T dy + diag(delta w) B dS
      dB = diag(delta) (L o Z)^T C + diag(delta w) x dS^T
      dC = diag(e^cum) dy S_in^T + (L o Z o delta_s) B
      dS_in = dec dS + C^T diag(e^cum) dy
    and for delta the gradient of the log-decays cum:
      dcum_t = row_t(F) - col_t(F) + e^(cum_t) dy_t . (C_t S_in) - w_t delta_t (B dS)_t . x_t
               (+ dS . S_out at the chunk's last step),  F = L o CB o Z o delta_s,
    ddelta_s = col_s(L o CB o Z) + w_s (B dS)_s . x_s + A sum_{t >= s} dcum_t,
    dA = sum_s delta_s sum_{t >= s} dcum_t (no delta limit here)."""
    x, Bm, Cm = p["x"], p["Bm"], p["Cm"]
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    hpg = H // G
    sarg = p["dt_raw"] + p["dt_bias"]
    delta = np.logaddexp(0.0, sarg)
    A = -np.exp(p["A_log"])
    r = {"dx": np.zeros_like(x), "ddt_raw": np.zeros_like(p["dt_raw"]), "ddt_bias": np.zeros(H),
         "dA_log": np.zeros(H), "dDp": np.zeros(H), "dBm": np.zeros_like(Bm), "dCm": np.zeros_like(Cm),
         "dh0": np.zeros_like(p["h0"])}
    for b in range(B):
        for h in range(H):
            g = h // hpg
            chunks = [(c0, min(L, c0 + Q)) for c0 in range(0, L, Q)]
            # forward: the state entering each chunk
            S = p["h0"][b, h].copy()
            S_in = []
            for c0, c1 in chunks:
                S_in.append(S.copy())
                dA_ = delta[b, c0:c1, h] * A[h]
                cum = np.cumsum(dA_)
                w = np.exp(cum[-1] - cum)
                S = np.exp(cum[-1]) * S + Bm[b, c0:c1, g].T @ ((w * delta[b, c0:c1, h])[:, None] * x[b, c0:c1, h])
            dS = dhl[b, h].copy()   # gradient of the state leaving the current chunk
            dA_h = 0.0
            for (c0, c1), Sin in reversed(list(zip(chunks, S_in))):
                dl = delta[b, c0:c1, h]
                cum = np.cumsum(dl * A[h])
                Lm = np.tril(np.exp(cum[:, None] - cum[None, :]))
                w = np.exp(cum[-1] - cum)
                dec = np.exp(cum[-1])
                xc, Bc, Cc, dyc = x[b, c0:c1, h], Bm[b, c0:c1, g], Cm[b, c0:c1, g], dy[b, c0:c1, h]
                CB = Cc @ Bc.T
                Z = dyc @ xc.T                       # Z[t][s] = dy_t . x_s
                Sout = dec * Sin + Bc.T @ ((w * dl)[:, None] * xc)
                BdS = Bc @ dS                        # [s][p]
                r["dx"][b, c0:c1, h] = p["Dp"][h] * dyc + dl[:, None] * ((Lm * CB).T @ dyc) + (dl * w)[:, None] * BdS
                r["dBm"][b, c0:c1, g] += dl[:, None] * ((Lm * Z).T @ Cc) + (dl * w)[:, None] * (xc @ dS.T)
                r["dCm"][b, c0:c1, g] += np.exp(cum)[:, None] * (dyc @ Sin.T) + (Lm * Z * dl[None, :]) @ Bc
                r["dDp"][h] += np.sum(dyc * xc)
                E = Lm * CB * Z                      # dloss/d(delta_s) through the intra term, before summing over t
                F = E * dl[None, :]
                R = np.exp(cum) * np.sum(dyc * (Cc @ Sin), axis=1)
                Wv = w * dl * np.sum(BdS * xc, axis=1)
                dcum = F.sum(axis=1) - F.sum(axis=0) + R - Wv
                dcum[-1] += np.sum(dS * Sout)
                direct = E.sum(axis=0) + w * np.sum(BdS * xc, axis=1)
                rev = np.cumsum(dcum[::-1])[::-1]    # sum over t >= i
                ddl = direct + A[h] * rev
                dA_h += np.sum(dl * rev)
                sig = 1.0 / (1.0 + np.exp(-sarg[b, c0:c1, h]))
                r["ddt_raw"][b, c0:c1, h] = ddl * sig
                dS = dec * dS + Cc.T @ (np.exp(cum)[:, None] * dyc)
            r["dh0"][b, h] = dS
            r["dA_log"][h] += dA_h * A[h]
    r["ddt_bias"] = r["ddt_raw"].sum(axis=(0, 1))
    return r


def check_bwd_chunked_form(seed=21, Q=4):
    p = _problem(B=2, L=13, H=4, P=3, G=2, N=3, seed=seed)
    r = np.random.default_rng(seed + 100)
    dy = r.standard_normal(p["x"].shape)
    dhl = r.standard_normal(p["h0"].shape)
    ref = oracle.ssd_bwd(*[p[k] for k in _KEYS], dy, dhl)
    got = chunked_backward(p, dy, dhl, Q)
    return max(float(np.max(np.abs(got[k] - ref[k])) / max(float(np.max(np.abs(ref[k]))), 1e-300)) for k in ref)


def check_bwd_finite_differences(dt_limit=None, seed=11):
    """Central differences (h = 1e-6) of loss = sum(dy*y) + sum(dh_last*h_last)
    against every gradient the backward returns; worst |fd - g| / max(1, |fd|)."""
    p = _problem(B=2, L=6, H=4, P=2, G=2, N=3, seed=seed)
    r = np.random.default_rng(seed + 100)
    dy = r.standard_normal(p["x"].shape)
    dhl = r.standard_normal(p["h0"].shape)
    lim = None
    if dt_limit == "quartiles":  # clamp about half the steps, at values no step sits on
        sp = np.logaddexp(0.0, p["dt_raw"] + p["dt_bias"]).ravel()
        lim = (float(np.quantile(sp, 0.25)) + 1e-3, float(np.quantile(sp, 0.75)) - 1e-3)

    def loss():
        y, hl = oracle.ssd_fwd(*[p[k] for k in _KEYS], dt_limit=lim)
        return float(np.sum(dy * y) + np.sum(dhl * hl))

    g = oracle.ssd_bwd(*[p[k] for k in _KEYS], dy, dhl, dt_limit=lim)
    worst, eps = 0.0, 1e-6
    for k in _KEYS:
        a = p[k]
        for idx in np.ndindex(a.shape):
            keep = a[idx]
            a[idx] = keep + eps
            lp = loss()
            a[idx] = keep - eps
            lm = loss()
            a[idx] = keep
            fd = (lp - lm) / (2 * eps)
            worst = max(worst, abs(fd - g[_GRAD[k]][idx]) / max(1.0, abs(fd)))
    return worst


def check_bwd_s6_reduction(dt_limit=None, seed=12):
    """The backward of each group equals the S6 oracle's backward of the
    mapped problem, summed over the head's P channels (delta, its bias, D),
    over P x N (A_log), and transposed (h0)."""
    p = _problem(seed=seed)
    B, L, H, P = p["x"].shape
    G, N = p["Bm"].shape[2], p["Bm"].shape[3]
    hpg = H // G
    r = np.random.default_rng(seed + 100)
    dy = r.standard_normal(p["x"].shape)
    dhl = r.standard_normal(p["h0"].shape)
    g = oracle.ssd_bwd(*[p[k] for k in _KEYS], dy, dhl, dt_limit=dt_limit)
    err = 0.0

    def rel(a, b):
        return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))

    for grp in range(G):
        hs = slice(grp * hpg, (grp + 1) * hpg)
        u = p["x"][:, :, hs, :].reshape(B, L, hpg * P)
        raw = np.repeat(p["dt_raw"][:, :, hs], P, axis=2)
        bias = np.repeat(p["dt_bias"][hs], P)
        A_log = np.repeat(p["A_log"][hs], P)[:, None] * np.ones((1, N))
        Dp = np.repeat(p["Dp"][hs], P)
        h0 = np.transpose(p["h0"][:, hs], (0, 1, 3, 2)).reshape(B, hpg * P, N)
        dout = dy[:, :, hs, :].reshape(B, L, hpg * P)
        dh_last = np.transpose(dhl[:, hs], (0, 1, 3, 2)).reshape(B, hpg * P, N)
        s6 = oracle.bwd(u, raw, None, p["Bm"][:, :, grp, :], p["Cm"][:, :, grp, :], A_log, Dp, bias, h0, dout,
                        dh_last, dt_limit=dt_limit)
        err = max(err, rel(g["dx"][:, :, hs, :], s6["du"].reshape(B, L, hpg, P)))
        err = max(err, rel(g["ddt_raw"][:, :, hs], s6["d_delta_raw"].reshape(B, L, hpg, P).sum(-1)))
        err = max(err, rel(g["ddt_bias"][hs], s6["d_delta_bias"].reshape(hpg, P).sum(-1)))
        err = max(err, rel(g["dA_log"][hs], s6["dA_log"].reshape(hpg, P, N).sum(axis=(1, 2))))
        err = max(err, rel(g["dDp"][hs], s6["dD"].reshape(hpg, P).sum(-1)))
        err = max(err, rel(g["dBm"][:, :, grp, :], s6["dBm"]))
        err = max(err, rel(g["dCm"][:, :, grp, :], s6["dCm"]))
        err = max(err, rel(g["dh0"][:, hs], np.transpose(s6["dh0"].reshape(B, hpg, P, N), (0, 1, 3, 2))))
    return err


PINS = {
    "s6_reduction": (lambda: check_s6_reduction(), 1e-12),
    "s6_reduction_limited": (lambda: check_s6_reduction(dt_limit=(0.3, 0.9), seed=3), 1e-12),
    "chunked_form": (lambda: check_chunked_form(), 1e-12),
    "chunked_form_q1": (lambda: check_chunked_form(seed=4, Q=1), 1e-12),
    "closed_form": (lambda: check_closed_form(), 1e-12),
    "dt_fixed_by_limit": (lambda: check_dt_fixed_by_limit(), 1e-12),
    "bwd_finite_differences": (lambda: check_bwd_finite_differences(), 1e-7),
    "bwd_finite_differences_limited": (lambda: check_bwd_finite_differences("quartiles", seed=13), 1e-7),
    "bwd_s6_reduction": (lambda: check_bwd_s6_reduction(), 1e-12),
    "bwd_chunked_form": (lambda: check_bwd_chunked_form(), 1e-12),
    "bwd_chunked_form_ragged": (lambda: check_bwd_chunked_form(seed=22, Q=5), 1e-12),
    "bwd_s6_reduction_limited": (lambda: check_bwd_s6_reduction(dt_limit=(0.3, 0.9), seed=14), 1e-12),
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_ssd_pin(name):
    fn, bound = PINS[name]
    err = fn()
    assert err <= bound, f"{name}: {err:.3e} > {bound:.1e}"


MUTANTS = {
    "group_index": ("const int64_t g = h / hpg;", "const int64_t g = h % G;"),
    "skip_dropped": ("yt[p] = acc + Dp[h] * xt[p];", "yt[p] = acc;"),
    "decay_sign": ("const double a = exp(delta * A);", "const double a = exp(-delta * A);"),
    "input_without_delta": ("delta * Bt[n] * xt[p];", "Bt[n] * xt[p];"),
    "B_for_C_readout": ("acc += Ct[n] * S[n * P + p];", "acc += Bt[n] * S[n * P + p];"),
    "bias_index": ("dt_raw[(b * L + t) * H + h] + dt_bias[h]", "dt_raw[(b * L + t) * H + h] + dt_bias[0]"),
    "dt_max_ignored": ("if (delta > dt_max) delta = dt_max;", ""),
    "readout_before_update": (
        "for (int64_t n = 0; n < N; ++n)\n          for (int64_t p = 0; p < P; ++p) S[n * P + p] = a * S[n * P + p] + delta * Bt[n] * xt[p];\n        double *yt",
        "double *yt"),
    "bwd_no_decay_of_adjoint": ("for (int64_t i = 0; i < NP; ++i) Gr[i] *= at;", ""),
    "bwd_dB_without_delta": ("dbv[n] += dl * sb;", "dbv[n] += sb;"),
    "bwd_ddelta_without_A": ("const double ddl = Ah * at * gs + gbx;", "const double ddl = at * gs + gbx;"),
    "bwd_dA_without_delta": ("dAh += dl * at * gs;", "dAh += at * gs;"),
    "bwd_limit_mask_ignored": ("(sp >= dt_min && sp <= dt_max) ? ddl * ssdo_sigmoid(sarg) : 0.0", "ddl * ssdo_sigmoid(sarg)"),
    "bwd_B_for_C_readout": ("Gr[n * P + p] += cv[n] * gy[p];", "Gr[n * P + p] += bv[n] * gy[p];"),
    "bwd_dx_skip_dropped": ("dxv[p] = Dp[h] * gy[p] + dl * sg;", "dxv[p] = dl * sg;"),
    "bwd_dh_last_ignored": ("if (dh_last)\n        memcpy(Gr,", "if (0)\n        memcpy(Gr,"),
    "bwd_dA_log_chain": ("dA_log[h] += dAh * Ah;", "dA_log[h] += dAh;"),
}


@pytest.mark.slow
@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_ssd_planted_mistake_is_caught(mutant, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")).read()
    old, new = MUTANTS[mutant]
    assert src.count(old) == 1, f"mutation anchor for {mutant} not found"
    cfile = tmp_path / "m.c"
    cfile.write_text(src.replace(old, new))
    so = oracle.build_ssd(force=True, src=str(cfile), out=str(tmp_path / "m.so"))
    failures = []
    with oracle.override_ssd_library(so):
        for name, (fn, bound) in PINS.items():
            if not (fn() <= bound):
                failures.append(name)
    assert failures, f"mutant {mutant} passed every pin"
