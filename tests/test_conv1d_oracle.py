"""Pins for the conv1d oracle (CPU only): an impulse response, numpy's own
convolution, central finite differences of every gradient, the single step
iterated against the multi-step forward (bit for bit), the state hand-over
between two halves of a sequence, and planted mistakes that must each fail a
pin."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

SILU = lambda v: v / (1.0 + np.exp(-v))  # noqa: E731


def _problem(B=2, L=9, D=3, K=4, seed=0, state=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, L, D))
    w = rng.standard_normal((D, K)) * 0.7
    bias = rng.standard_normal(D) * 0.3
    s0 = rng.standard_normal((B, D, K - 1)) if state else None
    dout = rng.standard_normal((B, L, D))
    return x, w, bias, s0, dout


def check_impulse():
    """A unit impulse at t0 (zero bias, zero state) puts tap K-1-j on output t0+j."""
    B, L, D, K, t0 = 1, 10, 2, 4, 3
    w = np.array([[0.5, -1.25, 2.0, 0.75], [1.5, 0.25, -0.5, 1.0]])
    x = np.zeros((B, L, D))
    x[0, t0, :] = 1.0
    out, _ = oracle.conv1d_fwd(x, w, np.zeros(D))
    want = np.zeros((B, L, D))
    for j in range(K):
        want[0, t0 + j, :] = SILU(w[:, K - 1 - j])
    return float(np.max(np.abs(out - want)))


def check_numpy_convolve():
    x, w, bias, s0, _ = _problem(B=2, L=11, D=3, K=4, seed=1)
    out, _ = oracle.conv1d_fwd(x, w, bias, s0)
    err = 0.0
    for b in range(x.shape[0]):
        for d in range(x.shape[2]):
            seq = np.concatenate([s0[b, d], x[b, :, d]])
            pre = bias[d] + np.convolve(seq, w[d][::-1], mode="valid")
            err = max(err, float(np.max(np.abs(out[b, :, d] - SILU(pre)))))
    return err


def _loss(x, w, bias, s0, dout):
    out, _ = oracle.conv1d_fwd(x, w, bias, s0)
    return float(np.sum(dout * out))


def check_finite_differences():
    x, w, bias, s0, dout = _problem(B=2, L=6, D=2, K=3, seed=2)
    g = oracle.conv1d_bwd(x, w, bias, s0, dout)
    worst = 0.0
    eps = 1e-6
    for name, arr, grad in (("x", x, g["dx"]), ("w", w, g["dw"]), ("bias", bias, g["dbias"]),
                            ("s0", s0, g["dstate0"])):
        for idx in np.ndindex(arr.shape):
            keep = arr[idx]
            arr[idx] = keep + eps
            lp = _loss(x, w, bias, s0, dout)
            arr[idx] = keep - eps
            lm = _loss(x, w, bias, s0, dout)
            arr[idx] = keep
            fd = (lp - lm) / (2 * eps)
            worst = max(worst, abs(fd - grad[idx]) / max(1.0, abs(fd)))
    return worst


def check_step_equals_scan():
    x, w, bias, s0, _ = _problem(B=2, L=8, D=3, K=4, seed=3)
    out, s_last = oracle.conv1d_fwd(x, w, bias, s0)
    st = s0.copy()
    err = 0.0
    for t in range(x.shape[1]):
        o, st = oracle.conv1d_step(x[:, t], w, bias, st)
        err = max(err, float(np.max(np.abs(o - out[:, t]))))
    return max(err, float(np.max(np.abs(st - s_last))))


def check_state_handover():
    """Two halves with the first half's final state equal the whole sequence."""
    x, w, bias, s0, _ = _problem(B=2, L=10, D=3, K=4, seed=4)
    out, s_last = oracle.conv1d_fwd(x, w, bias, s0)
    o1, s_mid = oracle.conv1d_fwd(x[:, :4], w, bias, s0)
    o2, s_end = oracle.conv1d_fwd(x[:, 4:], w, bias, s_mid)
    err = float(np.max(np.abs(np.concatenate([o1, o2], axis=1) - out)))
    return max(err, float(np.max(np.abs(s_end - s_last))))


PINS = {
    "impulse": (check_impulse, 1e-15),
    "numpy_convolve": (check_numpy_convolve, 1e-12),
    "finite_differences": (check_finite_differences, 1e-7),
    "step_equals_scan": (check_step_equals_scan, 0.0),
    "state_handover": (check_state_handover, 0.0),
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_conv1d_pin(name):
    fn, bound = PINS[name]
    err = fn()
    assert err <= bound, f"{name}: {err:.3e} > {bound:.1e}"


MUTANTS = {
    "taps_reversed": ("pre += w[d * K + k] * c1o_in(x, state0, L, D, K, b, t - (K - 1) + k, d);",
                      "pre += w[d * K + (K - 1 - k)] * c1o_in(x, state0, L, D, K, b, t - (K - 1) + k, d);"),
    "no_bias": ("double pre = bias[d];\n  for (int64_t k = 0; k < K; ++k)", "double pre = 0.0;\n  for (int64_t k = 0; k < K; ++k)"),
    "silu_derivative": ("s * (1.0 + pre * (1.0 - s))", "s * (1.0 + pre * s)"),
    "dx_shift": ("const int64_t to = t + (K - 1) - k;", "const int64_t to = t + K - k;"),
    "dw_offset": ("dw[d * K + k] += g * c1o_in(x, state0, L, D, K, b, t - (K - 1) + k, d);",
                  "dw[d * K + k] += g * c1o_in(x, state0, L, D, K, b, t - K + k, d);"),
    "dstate_offset": ("const int64_t to = j - k;", "const int64_t to = j - k + 1;"),
    "state_oldest_last": ("return state0[(b * D + d) * (K - 1) + (K - 1 + t)];", "return state0[(b * D + d) * (K - 1) + (-1 - t)];"),
    "step_no_shift": ("for (int64_t k = 0; k + 1 < K - 1; ++k) st[k] = st[k + 1];", "for (int64_t k = 0; k + 1 < K - 1; ++k) st[k] = st[k];"),
}


@pytest.mark.slow
@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_conv1d_planted_mistake_is_caught(mutant, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "conv1d_oracle.c")).read()
    old, new = MUTANTS[mutant]
    assert src.count(old) == 1, f"mutation anchor for {mutant} not found"
    cfile = tmp_path / "m.c"
    cfile.write_text(src.replace(old, new))
    so = oracle.build_conv1d(force=True, src=str(cfile), out=str(tmp_path / "m.so"))
    failures = []
    with oracle.override_conv1d_library(so):
        for name, (fn, bound) in PINS.items():
            if not (fn() <= bound):
                failures.append(name)
    assert failures, f"mutant {mutant} passed every pin"
