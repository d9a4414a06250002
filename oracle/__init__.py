"""Oracle for the S6 selective scan: plain f64 CPU reference (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library in
``selective_state_space_s6_gb300``) never imports it, and it imports nothing
from there.

The arithmetic lives in ``ssm_oracle.c`` (plain sequential C, f64); this
module only compiles it with gcc (``build()``) and marshals numpy arrays.
What it computes, and which page each step follows, is in that file's header:
the recurrence, discretisation and readout of the final selective_scan_kernel
on the POPCORNBENCH transcript page (FW-GLM-5-1__l2_p30), with the softplus,
exp_negate, SiLU-gate and gating-backward steps named by the mamba-rs
kernels.rs page (MambaKernels doc comments), and a chain-rule backward that no
page writes out (pinned in tests by finite differences).  The optional limit
on Δ (``dt_limit``) is the clamp and gradient mask of the
mamba3_preprocess_backward.slang page.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libssm_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ssm_oracle.c`` into ``_build/libssm_oracle.so`` (gcc, -O2, pthreads)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-adds, so every product and sum is
    # rounded exactly as written; the oracle stays a literal reading of the math.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _open(path):
    lib = ctypes.CDLL(path)
    i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    f64 = ctypes.c_double
    lib.s6o_fwd.argtypes = [i64] * 4 + [vp] * 9 + [vp] * 2 + [i64] * 4 + [ci, f64, f64]
    lib.s6o_fwd.restype = ci
    lib.s6o_bwd.argtypes = [i64] * 4 + [vp] * 9 + [vp] * 2 + [vp] * 9 + [i64] * 4 + [ci, f64, f64]
    lib.s6o_bwd.restype = ci
    lib.s6o_step.argtypes = [i64] * 3 + [vp] * 8 + [vp] * 2 + [f64, f64]
    lib.s6o_step.restype = ci
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(build())
    return _lib


@contextlib.contextmanager
def override_library(path):
    """Run the wrappers against another build of the oracle source (used by the
    tests that plant a mistake in a copy of ``ssm_oracle.c``)."""
    global _lib
    prev = _load()
    with _lock:
        _lib = _open(path)
    try:
        yield
    finally:
        with _lock:
            _lib = prev


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen exactly (bf16/f32 -> f64)
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _limits(dt_limit):
    """(dt_min, dt_max) of the Δ clamp; None means no limit, (0, +inf)."""
    if dt_limit is None:
        return 0.0, float("inf")
    lo, hi = float(dt_limit[0]), float(dt_limit[1])
    return lo, hi


def _shapes(u, Bm):
    B, L, D = u.shape
    N = Bm.shape[2]
    return B, L, D, N


def fwd(u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h0=None, *, b_range=None,
        d_range=None, threads=None, dt_limit=None):
    """Forward scan.  Returns ``(out [B,L,D], h_last [B,D,N])`` as f64 arrays.

    With ``b_range``/``d_range`` only those batches/channels are computed; the
    other entries of the returned arrays are NaN.  ``dt_limit = (dt_min,
    dt_max)`` clamps Δ = softplus(s) to that range.
    """
    u, delta_raw, z, Bm, Cm = map(_f64, (u, delta_raw, z, Bm, Cm))
    A_log, Dp, delta_bias, h0 = map(_f64, (A_log, Dp, delta_bias, h0))
    B, L, D, N = _shapes(u, Bm)
    b0, b1 = b_range or (0, B)
    d0, d1 = d_range or (0, D)
    out = np.full((B, L, D), np.nan)
    h_last = np.full((B, D, N), np.nan)
    rc = _load().s6o_fwd(B, L, D, N, _ptr(u), _ptr(delta_raw), _ptr(z), _ptr(Bm), _ptr(Cm),
                         _ptr(A_log), _ptr(Dp), _ptr(delta_bias), _ptr(h0), _ptr(out),
                         _ptr(h_last), b0, b1, d0, d1, threads or default_threads(), *_limits(dt_limit))
    if rc != 0:
        raise ValueError(f"s6o_fwd failed with code {rc}")
    return out, h_last


def bwd(u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h0, dout, dh_last=None, *,
        b_range=None, d_range=None, threads=None, dt_limit=None):
    """Backward of ``loss = sum(dout*out) + sum(dh_last*h_last)``.

    Returns a dict of f64 arrays: du, d_delta_raw, dz (NaN where not computed),
    dBm, dCm (sums over the selected channels), dA_log, dD, d_delta_bias (sums
    over the selected batches), dh0.
    """
    u, delta_raw, z, Bm, Cm = map(_f64, (u, delta_raw, z, Bm, Cm))
    A_log, Dp, delta_bias, h0, dout, dh_last = map(_f64, (A_log, Dp, delta_bias, h0, dout, dh_last))
    B, L, D, N = _shapes(u, Bm)
    b0, b1 = b_range or (0, B)
    d0, d1 = d_range or (0, D)
    r = {
        "du": np.full((B, L, D), np.nan), "d_delta_raw": np.full((B, L, D), np.nan),
        "dz": np.full((B, L, D), np.nan) if z is not None else None,
        "dBm": np.zeros((B, L, N)), "dCm": np.zeros((B, L, N)),
        "dA_log": np.full((D, N), np.nan), "dD": np.full((D,), np.nan),
        "d_delta_bias": np.full((D,), np.nan), "dh0": np.full((B, D, N), np.nan),
    }
    rc = _load().s6o_bwd(B, L, D, N, _ptr(u), _ptr(delta_raw), _ptr(z), _ptr(Bm), _ptr(Cm),
                         _ptr(A_log), _ptr(Dp), _ptr(delta_bias), _ptr(h0), _ptr(dout),
                         _ptr(dh_last), _ptr(r["du"]), _ptr(r["d_delta_raw"]), _ptr(r["dz"]),
                         _ptr(r["dBm"]), _ptr(r["dCm"]), _ptr(r["dA_log"]), _ptr(r["dD"]),
                         _ptr(r["d_delta_bias"]), _ptr(r["dh0"]), b0, b1, d0, d1,
                         threads or default_threads(), *_limits(dt_limit))
    if rc != 0:
        raise ValueError(f"s6o_bwd failed with code {rc}")
    return r


def step(u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h, *, dt_limit=None):
    """One decode step (T = 1).  u, delta_raw, z: [B,D]; Bm, Cm: [B,N]; h: [B,D,N].

    Returns ``(out [B,D], h_new [B,D,N])``; the input ``h`` is not modified.
    """
    u, delta_raw, z, Bm, Cm = map(_f64, (u, delta_raw, z, Bm, Cm))
    A_log, Dp, delta_bias = map(_f64, (A_log, Dp, delta_bias))
    h_new = _f64(h).copy()
    B, D = u.shape
    N = Bm.shape[1]
    out = np.full((B, D), np.nan)
    rc = _load().s6o_step(B, D, N, _ptr(u), _ptr(delta_raw), _ptr(z), _ptr(Bm), _ptr(Cm),
                          _ptr(A_log), _ptr(Dp), _ptr(delta_bias), _ptr(h_new), _ptr(out),
                          *_limits(dt_limit))
    if rc != 0:
        raise ValueError(f"s6o_step failed with code {rc}")
    return out, h_new


# ------------------------------------------------------------------ conv1d
# The causal depthwise conv1d + SiLU in front of the scan: ``conv1d_oracle.c``
# (plain sequential C, f64), built into its own library.

_CONV_SRC = os.path.join(_HERE, "conv1d_oracle.c")
_CONV_LIB_PATH = os.path.join(_BUILD_DIR, "libconv1d_oracle.so")
_conv_lib = None


def build_conv1d(force: bool = False, src: str = None, out: str = None) -> str:
    """Compile ``conv1d_oracle.c`` (or ``src``) into a shared library (gcc, -O2)."""
    src = src or _CONV_SRC
    out = out or _CONV_LIB_PATH
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                    "-Wall", "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _open_conv(path):
    lib = ctypes.CDLL(path)
    i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.c1o_fwd.argtypes = [i64] * 4 + [vp] * 6
    lib.c1o_fwd.restype = ci
    lib.c1o_bwd.argtypes = [i64] * 4 + [vp] * 9
    lib.c1o_bwd.restype = ci
    lib.c1o_step.argtypes = [i64] * 3 + [vp] * 5
    lib.c1o_step.restype = ci
    return lib


def _load_conv():
    global _conv_lib
    with _lock:
        if _conv_lib is None:
            _conv_lib = _open_conv(build_conv1d())
    return _conv_lib


@contextlib.contextmanager
def override_conv1d_library(path):
    """Run the conv1d wrappers against another build (planted-mistake tests)."""
    global _conv_lib
    prev = _load_conv()
    with _lock:
        _conv_lib = _open_conv(path)
    try:
        yield
    finally:
        with _lock:
            _conv_lib = prev


def conv1d_fwd(x, w, bias, state0=None):
    """Causal depthwise conv1d + SiLU.  x [B,L,D], w [D,K], bias [D], state0
    [B,D,K-1] (the K-1 inputs before t = 0; zeros when None).  Returns
    ``(out [B,L,D], state_last [B,D,K-1])`` as f64 arrays."""
    x, w, bias, state0 = map(_f64, (x, w, bias, state0))
    B, L, D = x.shape
    K = w.shape[1]
    out = np.full((B, L, D), np.nan)
    state_last = np.full((B, D, max(K - 1, 0)), np.nan)
    rc = _load_conv().c1o_fwd(B, L, D, K, _ptr(x), _ptr(w), _ptr(bias), _ptr(state0), _ptr(out),
                              _ptr(state_last))
    if rc != 0:
        raise ValueError(f"c1o_fwd failed with code {rc}")
    return out, state_last


def conv1d_bwd(x, w, bias, state0, dout):
    """Backward of ``loss = sum(dout * out)``: dict of f64 arrays dx, dw, dbias, dstate0."""
    x, w, bias, state0, dout = map(_f64, (x, w, bias, state0, dout))
    B, L, D = x.shape
    K = w.shape[1]
    r = {"dx": np.full((B, L, D), np.nan), "dw": np.full((D, K), np.nan), "dbias": np.full((D,), np.nan),
         "dstate0": np.full((B, D, max(K - 1, 0)), np.nan)}
    rc = _load_conv().c1o_bwd(B, L, D, K, _ptr(x), _ptr(w), _ptr(bias), _ptr(state0), _ptr(dout),
                              _ptr(r["dx"]), _ptr(r["dw"]), _ptr(r["dbias"]), _ptr(r["dstate0"]))
    if rc != 0:
        raise ValueError(f"c1o_bwd failed with code {rc}")
    return r


def conv1d_step(x_t, w, bias, state):
    """One step: x_t [B,D], state [B,D,K-1] (not modified).  Returns ``(out [B,D], state_new)``."""
    x_t, w, bias = map(_f64, (x_t, w, bias))
    st = _f64(state).copy()
    B, D = x_t.shape
    K = w.shape[1]
    out = np.full((B, D), np.nan)
    rc = _load_conv().c1o_step(B, D, K, _ptr(x_t), _ptr(w), _ptr(bias), _ptr(st), _ptr(out))
    if rc != 0:
        raise ValueError(f"c1o_step failed with code {rc}")
    return out, st


# ------------------------------------------------------------------ Mamba-2 SSD
# The scalar-A-per-head variant of the scan (``ssd_oracle.c``, plain
# sequential C, f64), built into its own library.

_SSD_SRC = os.path.join(_HERE, "ssd_oracle.c")
_SSD_LIB_PATH = os.path.join(_BUILD_DIR, "libssd_oracle.so")
_ssd_lib = None


def build_ssd(force: bool = False, src: str = None, out: str = None) -> str:
    """Compile ``ssd_oracle.c`` (or ``src``) into a shared library (gcc, -O2)."""
    src = src or _SSD_SRC
    out = out or _SSD_LIB_PATH
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                    "-Wall", "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _open_ssd(path):
    lib = ctypes.CDLL(path)
    i64, vp, ci, f64 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.ssdo_fwd.argtypes = [i64] * 6 + [vp] * 8 + [f64, f64] + [vp] * 2
    lib.ssdo_fwd.restype = ci
    lib.ssdo_bwd.argtypes = [i64] * 6 + [vp] * 10 + [f64, f64] + [vp] * 8
    lib.ssdo_bwd.restype = ci
    return lib


def _load_ssd():
    global _ssd_lib
    with _lock:
        if _ssd_lib is None:
            _ssd_lib = _open_ssd(build_ssd())
    return _ssd_lib


@contextlib.contextmanager
def override_ssd_library(path):
    """Run the SSD wrapper against another build (planted-mistake tests)."""
    global _ssd_lib
    prev = _load_ssd()
    with _lock:
        _ssd_lib = _open_ssd(path)
    try:
        yield
    finally:
        with _lock:
            _ssd_lib = prev


def ssd_fwd(x, dt_raw, dt_bias, A_log, Bm, Cm, Dp, h0=None, *, dt_limit=None):
    """Mamba-2 SSD forward, step by step.  x [B,L,H,P], dt_raw [B,L,H], dt_bias /
    A_log / Dp [H], Bm / Cm [B,L,G,N], h0 [B,H,N,P] (zeros when None).  Returns
    ``(y [B,L,H,P], h_last [B,H,N,P])`` as f64 arrays."""
    x, dt_raw, dt_bias, A_log, Bm, Cm, Dp, h0 = map(_f64, (x, dt_raw, dt_bias, A_log, Bm, Cm, Dp, h0))
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    y = np.full((B, L, H, P), np.nan)
    h_last = np.full((B, H, N, P), np.nan)
    rc = _load_ssd().ssdo_fwd(B, L, H, P, G, N, _ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(A_log), _ptr(Bm),
                              _ptr(Cm), _ptr(Dp), _ptr(h0), *_limits(dt_limit), _ptr(y), _ptr(h_last))
    if rc != 0:
        raise ValueError(f"ssdo_fwd failed with code {rc}")
    return y, h_last


def ssd_bwd(x, dt_raw, dt_bias, A_log, Bm, Cm, Dp, h0, dy, dh_last=None, *, dt_limit=None):
    """Backward of ``loss = sum(dy*y) + sum(dh_last*h_last)`` through the SSD
    recurrence, step by step.  Returns a dict of f64 arrays: dx [B,L,H,P],
    ddt_raw [B,L,H], ddt_bias / dA_log / dDp [H] (sums over batch and steps),
    dBm / dCm [B,L,G,N] (sums over the heads of a group), dh0 [B,H,N,P]."""
    x, dt_raw, dt_bias, A_log, Bm, Cm, Dp, h0, dy, dh_last = map(
        _f64, (x, dt_raw, dt_bias, A_log, Bm, Cm, Dp, h0, dy, dh_last))
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    r = {"dx": np.full((B, L, H, P), np.nan), "ddt_raw": np.full((B, L, H), np.nan),
         "ddt_bias": np.full((H,), np.nan), "dA_log": np.full((H,), np.nan), "dDp": np.full((H,), np.nan),
         "dBm": np.full((B, L, G, N), np.nan), "dCm": np.full((B, L, G, N), np.nan),
         "dh0": np.full((B, H, N, P), np.nan)}
    rc = _load_ssd().ssdo_bwd(B, L, H, P, G, N, _ptr(x), _ptr(dt_raw), _ptr(dt_bias), _ptr(A_log), _ptr(Bm),
                              _ptr(Cm), _ptr(Dp), _ptr(h0), _ptr(dy), _ptr(dh_last), *_limits(dt_limit),
                              _ptr(r["dx"]), _ptr(r["ddt_raw"]), _ptr(r["ddt_bias"]), _ptr(r["dA_log"]),
                              _ptr(r["dBm"]), _ptr(r["dCm"]), _ptr(r["dDp"]), _ptr(r["dh0"]))
    if rc != 0:
        raise ValueError(f"ssdo_bwd failed with code {rc}")
    return r
