"""Pins for the f64 oracle (CPU only).

The oracle is trusted only because these checks tie it to things other than
itself: a non-recursive closed form, central finite differences, textbook
special cases, limits, invariants and a hand-worked example.
"""
import json
import os
import shutil
import subprocess

import numpy as np
import pytest
from scipy.special import expit

import oracle
import oracle_checks as oc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("name", sorted(oc.ALL_CHECKS))
def test_pin(name):
    fn, bound = oc.ALL_CHECKS[name]
    err = fn()
    assert err <= bound, f"{name}: error {err:.3e} > {bound:.1e}"


def test_hand_worked_golden():
    with open(os.path.join(GOLDEN, "hand_worked_l2.json")) as f:
        fx = json.load(f)
    assert oc.check_hand_worked(fx) <= fx["tolerance_abs"]


def test_single_cell_by_hand():
    """N=1, L=1: y = C Δ B u + D u, out = y z σ(z)."""
    u, raw, bias, B, C, Dp, z, A_log = 0.9, -0.3, 0.1, 1.7, -0.4, 0.6, 1.3, 0.2
    delta = np.log1p(np.exp(raw + bias))
    y = C * delta * B * u + Dp * u
    out, h_last = oracle.fwd(np.array([[[u]]]), np.array([[[raw]]]), np.array([[[z]]]),
                             np.array([[[B]]]), np.array([[[C]]]), np.array([[A_log]]),
                             np.array([Dp]), np.array([bias]))
    assert abs(out[0, 0, 0] - y * z * expit(z)) < 1e-15
    assert abs(h_last[0, 0, 0] - delta * B * u) < 1e-15


def test_step_iterated_equals_scan_bitwise():
    p, _, _ = oc.rand_problem(2, 11, 3, 4, seed=7)
    out, h_last = oracle.fwd(p["u"], p["delta_raw"], p["z"], p["Bm"], p["Cm"], p["A_log"],
                             p["Dp"], p["delta_bias"], p["h0"])
    h = p["h0"].copy()
    for t in range(p["u"].shape[1]):
        o, h = oracle.step(p["u"][:, t], p["delta_raw"][:, t], p["z"][:, t], p["Bm"][:, t],
                           p["Cm"][:, t], p["A_log"], p["Dp"], p["delta_bias"], h)
        assert np.array_equal(o, out[:, t])
    assert np.array_equal(h, h_last)


def test_linear_in_u_and_h0():
    p1, _, _ = oc.rand_problem(2, 9, 3, 4, seed=8)
    p2, _, _ = oc.rand_problem(2, 9, 3, 4, seed=9)
    alpha, beta = 0.7, -1.3
    base = dict(p1)
    mix = dict(p1)
    mix["u"] = alpha * p1["u"] + beta * p2["u"]
    mix["h0"] = alpha * p1["h0"] + beta * p2["h0"]
    other = dict(p1)
    other["u"], other["h0"] = p2["u"], p2["h0"]
    args = ("u", "delta_raw", "z", "Bm", "Cm", "A_log", "Dp", "delta_bias", "h0")
    o1, h1 = oracle.fwd(*[base[k] for k in args])
    o2, h2 = oracle.fwd(*[other[k] for k in args])
    om, hm = oracle.fwd(*[mix[k] for k in args])
    assert np.max(np.abs(om - (alpha * o1 + beta * o2))) < 1e-12 * np.max(np.abs(om))
    assert np.max(np.abs(hm - (alpha * h1 + beta * h2))) < 1e-12 * np.max(np.abs(hm))


def test_causal():
    p, _, _ = oc.rand_problem(1, 12, 3, 4, seed=10)
    args = ("u", "delta_raw", "z", "Bm", "Cm", "A_log", "Dp", "delta_bias", "h0")
    o1, _ = oracle.fwd(*[p[k] for k in args])
    t0 = 6
    for key in ("u", "delta_raw", "Bm", "Cm", "z"):
        q = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
        q[key][:, t0] += 1.0
        o2, _ = oracle.fwd(*[q[k] for k in args])
        assert np.array_equal(o1[:, :t0], o2[:, :t0]), key
        assert not np.array_equal(o1[:, t0], o2[:, t0]), key


def test_subranges_match_full_run():
    """Channel/batch sub-ranges (used for sampled checks at full size) agree with the
    full run; dBm/dCm over a partition of channels add up to the full sums."""
    p, dout, dh_last = oc.rand_problem(3, 10, 70, 3, seed=11)
    args = [p[k] for k in ("u", "delta_raw", "z", "Bm", "Cm", "A_log", "Dp", "delta_bias", "h0")]
    full = oracle.bwd(*args, dout, dh_last)
    fo, fh = oracle.fwd(*args)
    so, sh = oracle.fwd(*args, b_range=(1, 2), d_range=(5, 9))
    assert np.array_equal(so[1, :, 5:9], fo[1, :, 5:9])
    assert np.array_equal(sh[1, 5:9], fh[1, 5:9])
    parts = [oracle.bwd(*args, dout, dh_last, d_range=r) for r in ((0, 20), (20, 64), (64, 70))]
    for key in ("dBm", "dCm"):
        tot = sum(pt[key] for pt in parts)
        assert np.max(np.abs(tot - full[key])) < 1e-12 * np.max(np.abs(full[key]))
    sub = oracle.bwd(*args, dout, dh_last, d_range=(5, 9))
    for key in ("du", "d_delta_raw", "dz"):
        assert np.array_equal(sub[key][:, :, 5:9], full[key][:, :, 5:9])
    for key in ("dA_log", "dD", "d_delta_bias"):
        assert np.array_equal(sub[key][5:9], full[key][5:9])


def test_thread_count_invariant():
    p, dout, dh_last = oc.rand_problem(2, 9, 150, 3, seed=12)
    args = [p[k] for k in ("u", "delta_raw", "z", "Bm", "Cm", "A_log", "Dp", "delta_bias", "h0")]
    a = oracle.bwd(*args, dout, dh_last, threads=1)
    b = oracle.bwd(*args, dout, dh_last, threads=5)
    for k in a:
        if a[k] is not None:
            assert np.array_equal(a[k], b[k]), k


# --------------------------------------------------------------- planted mistakes

# Each mutant is a plausible slip in the oracle source; at least one pin must catch it.
MUTANTS = {
    "drop_skip": ("y += p->Dp[d] * u;", "y += 0.0 * u;"),
    "decay_sign": ("const double a = exp(delta * A);", "const double a = exp(-delta * A);"),
    "B_for_C_readout": ("y += p->Cm[ix_bln(p, b, t, n)] * h[n];", "y += p->Bm[ix_bln(p, b, t, n)] * h[n];"),
    "drop_delta_in_input": ("const double bt = delta * p->Bm[ix_bln(p, b, t, n)] * u;",
                            "const double bt = p->Bm[ix_bln(p, b, t, n)] * u;"),
    "softplus_branch": ("s + log1p(exp(-s))", "log1p(exp(-s))"),
    "gate_without_z": ("o = y * z * s6o_sigmoid(z);", "o = y * s6o_sigmoid(z);"),
    "bias_index": ("p->delta_bias[d];\n    const double delta = s6o_delta(p, s6o_softplus(s));\n    double y",
                   "p->delta_bias[0];\n    const double delta = s6o_delta(p, s6o_softplus(s));\n    double y"),
    "dz_formula": ("(1.0 + z * (1.0 - sz))", "(1.0 + z * sz)"),
    "g_no_decay": ("g[n] = a * gt;", "g[n] = gt;"),
    "ddelta_drop_state_term": ("gt * (A * a * h_prev + Bn * u)", "gt * (Bn * u)"),
    "dA_log_missing_A": ("-exp(p->A_log[d * N + n]) * acc_dA[n]", "acc_dA[n]"),
    "du_uses_dout": ("p->Dp[d] * dy + delta * sum_gB", "p->Dp[d] * dout + delta * sum_gB"),
    "d_raw_wrong_sigmoid": ("sum_dh_ddelta * s6o_sigmoid(s)", "sum_dh_ddelta * s6o_sigmoid(-s)"),
    "dC_uses_h_prev": ("dy * hist_h[t * N + n]", "dy * h_prev"),
    "dB_drops_delta": ("pdB[t * N + n] += gt * delta * u;", "pdB[t * N + n] += gt * u;"),
    "h_prev_off_by_one": ("hist_h[(t - 1) * N + n]", "hist_h[t * N + n]"),
    "dh_last_ignored": ("g[n] = job->dh_last ? job->dh_last[(b * p->D + d) * N + n] : 0.0;",
                        "g[n] = 0.0;"),
    "dt_mask_dropped": ("sum_dh_ddelta * s6o_sigmoid(s) * mask", "sum_dh_ddelta * s6o_sigmoid(s)"),
    "dt_mask_inverted": ("? 1.0 : 0.0;", "? 0.0 : 1.0;"),
    "dt_clamp_on_s": ("const double delta = s6o_delta(p, s6o_softplus(s));",
                      "const double delta = s6o_softplus(s6o_delta(p, s));"),
    "dt_max_ignored": ("if (sp > p->dt_max) return p->dt_max;", ""),
    "dt_bwd_unclamped_delta": ("const double delta = s6o_delta(p, sp);", "const double delta = sp;"),
}


@pytest.mark.slow
@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")).read()
    old, new = MUTANTS[mutant]
    assert src.count(old) >= 1, f"mutation anchor for {mutant} not found"
    mutated = src.replace(old, new, 1)
    cfile = tmp_path / "m.c"
    cfile.write_text(mutated)
    so = tmp_path / "m.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    "-o", str(so), str(cfile), "-lm"], check=True)
    with open(os.path.join(GOLDEN, "hand_worked_l2.json")) as f:
        fx = json.load(f)
    failures = []
    with oracle.override_library(str(so)):
        for name, (fn, bound) in oc.ALL_CHECKS.items():
            err = fn()
            if not (err <= bound):
                failures.append(name)
        if not (oc.check_hand_worked(fx) <= fx["tolerance_abs"]):
            failures.append("hand_worked")
    assert failures, f"mutant {mutant} passed every pin"
