"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
(via the Python binding) and compare with the oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from selective_state_space_s6_gb300 import s6

# Tolerances: max relative error, normwise per output tensor
#   max_i |gpu_i - oracle_i| / max_i |oracle_i|
# fp32 I/O: 1e-5; bf16 I/O with f32 state and arithmetic: 2e-2.
TOL = {"f32": 1e-5, "bf16": 2e-2}

ARGS = ("u", "delta_raw", "z", "Bm", "Cm", "A_log", "Dp", "delta_bias")


def to_dev(x, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def act_of(x):
    return "bf16" if x["u"].dtype == torch.bfloat16 else "f32"


def np64(t):
    return None if t is None else t.detach().to("cpu").double().numpy()


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0
    assert np.all(np.isfinite(got)), "non-finite values in GPU output"
    scale = np.max(np.abs(ref))
    diff = np.max(np.abs(got - ref))
    return float(diff / scale) if scale > 0 else float(diff)


def gpu_fwd_bwd(xd, dh_last=None, want_bwd=True, dt_limit=None):
    """Run the CUDA path on device inputs ``xd``; returns dict of torch tensors."""
    out, h_last, cs = s6.ssm_scan_fwd(*[xd[k] for k in ARGS], xd.get("h0"), dt_limit=dt_limit)
    r = {"out": out, "h_last": h_last, "chunk_states": cs}
    if want_bwd:
        g = s6.ssm_scan_bwd(*[xd[k] for k in ARGS], xd.get("h0"), cs, xd["dout"], dh_last,
                            dt_limit=dt_limit)
        r.update(g)
    s6.check_device_status()  # synchronises; raises if a bounded device wait gave up
    return r


def oracle_fwd_bwd(x, dh_last=None, want_bwd=True, **kw):
    out, h_last = oracle.fwd(*[x[k] for k in ARGS], x.get("h0"), **kw)
    r = {"out": out, "h_last": h_last}
    if want_bwd:
        r.update(oracle.bwd(*[x[k] for k in ARGS], x.get("h0"), x["dout"], dh_last, **kw))
    return r


GRAD_KEYS = ("du", "d_delta_raw", "dz", "dBm", "dCm", "dA_log", "dD", "d_delta_bias", "dh0")


def compare_all(gpu, ref, tol, keys=("out", "h_last") + GRAD_KEYS):
    errs = {}
    for k in keys:
        if ref.get(k) is None or gpu.get(k) is None:
            continue
        errs[k] = rel_err(np64(gpu[k]), ref[k])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"errors above {tol}: {bad} (all: {errs})"
    return errs
