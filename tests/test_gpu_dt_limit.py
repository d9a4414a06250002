"""The limit on delta (dt_limit: delta = clamp(softplus(s), dt_min, dt_max),
no gradient to delta_raw / delta_bias through a clamped step) on the GPU,
through the C ABI's _ex entry points, against the f64 oracle with the same
limit: forward, backward, the decode step (iterated, bit for bit against the
scan), and the plain calls reproduced exactly by the _ex calls with no limit.

Inputs: the seeded generator's, with [dt_min, dt_max] at the 25% / 75%
quantiles of the drawn softplus(s) so that both ends clamp about a quarter
of the steps; any delta_raw whose softplus lies within 0.2% of a bound is
moved off it (an f32 softplus and the f64 one must fall on the same side)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import ARGS, TOL, compare_all, gpu_fwd_bwd, np64, oracle_fwd_bwd, to_dev
from selective_state_space_s6_gb300 import inputs, s6

pytestmark = pytest.mark.gpu


def limited_problem(B, L, D, N, act, seed, lo_q=0.25, hi_q=0.75, margin=2e-3):
    x = inputs.make_inputs(B, L, D, N, act, seed=seed, h0_std=0.5, with_dh_last=True)
    dt = x["delta_raw"].dtype

    def softplus():
        s = x["delta_raw"].double() + x["delta_bias"].double()
        return torch.nn.functional.softplus(s)

    sp = softplus().numpy().reshape(-1)
    sample = sp[:: max(1, sp.size // 200000)]
    lo, hi = float(np.quantile(sample, lo_q)), float(np.quantile(sample, hi_q))
    lo, hi = float(np.float32(lo)), float(np.float32(hi))  # the values the GPU is given
    for _ in range(20):
        sp = softplus()
        near = ((sp - lo).abs() < margin * lo) | ((sp - hi).abs() < margin * hi)
        if not bool(near.any()):
            return x, (lo, hi)
        raw = x["delta_raw"].double()
        raw[near] += 0.05
        x["delta_raw"] = raw.to(dt)
    raise AssertionError("could not move the inputs off the bounds")


SHAPES = [
    (2, 300, 128, 16, "bf16"),   # TMA scan
    (2, 200, 96, 16, "f32"),
    (3, 130, 64, 8, "bf16"),
    (1, 3000, 64, 16, "f32"),    # long sequence, few channels: time split across CTAs
    (2, 100, 40, 5, "f32"),      # N = 5: the generic kernels
]


@pytest.mark.parametrize("B,L,D,N,act", SHAPES)
def test_dt_limit_parity(B, L, D, N, act):
    x, lim = limited_problem(B, L, D, N, act, seed=B + L + N)
    xd = to_dev(x)
    gpu = gpu_fwd_bwd(xd, dh_last=xd["dh_last"], dt_limit=lim)
    ref = oracle_fwd_bwd(x, dh_last=x["dh_last"], dt_limit=lim)
    # the limit is active: a quarter of the steps pass no gradient to delta_raw
    zero = np.mean(ref["d_delta_raw"] == 0.0)
    assert 0.3 < zero < 0.7, zero
    compare_all(gpu, ref, TOL[act])
    # and the GPU zeroes exactly the steps the oracle zeroes
    assert np.array_equal(np64(gpu["d_delta_raw"]) == 0.0, ref["d_delta_raw"] == 0.0)


@pytest.mark.parametrize("act", ["f32", "bf16"])
def test_dt_limit_step_chain_equals_scan_bitwise(act):
    B, L, D, N = 4, 24, 64, 16
    x, lim = limited_problem(B, L, D, N, act, seed=3)
    xd = to_dev(x)
    out, h_last, _ = s6.ssm_scan_fwd(*[xd[k] for k in ARGS], xd["h0"], dt_limit=lim)
    h = xd["h0"].clone()
    for t in range(L):
        o = s6.ssm_step(*[xd[k][:, t].contiguous() if k in ("u", "delta_raw", "z", "Bm", "Cm") else xd[k]
                          for k in ARGS], h, dt_limit=lim)
        assert torch.equal(o, out[:, t]), t
    assert torch.equal(h, h_last)
    ref_o, ref_h = oracle.step(*[x[k][:, 0] if k in ("u", "delta_raw", "z", "Bm", "Cm") else x[k]
                                 for k in ARGS], x["h0"], dt_limit=lim)
    o0 = s6.ssm_step(*[xd[k][:, 0].contiguous() if k in ("u", "delta_raw", "z", "Bm", "Cm") else xd[k]
                       for k in ARGS], xd["h0"].clone(), dt_limit=lim)
    assert np.max(np.abs(np64(o0) - ref_o)) / np.max(np.abs(ref_o)) <= TOL[act]


@pytest.mark.parametrize("act", ["f32", "bf16"])
def test_no_limit_equals_plain_calls_bitwise(act):
    x = inputs.make_inputs(2, 333, 128, 16, act, seed=9, h0_std=0.5, with_dh_last=True)
    xd = to_dev(x)
    plain = gpu_fwd_bwd(xd, dh_last=xd["dh_last"])
    ex = gpu_fwd_bwd(xd, dh_last=xd["dh_last"], dt_limit=(0.0, float("inf")))
    for k, v in plain.items():
        if v is not None:
            assert torch.equal(v, ex[k]), k


def test_bad_limit_is_rejected():
    x = to_dev(inputs.make_inputs(1, 8, 16, 4, "f32", seed=1))
    for lim in ((0.5, 0.1), (-1.0, 1.0), (float("nan"), 1.0)):
        with pytest.raises(s6.SSMError) as err:
            s6.ssm_scan_fwd(*[x[k] for k in ARGS], None, dt_limit=lim)
        assert "SSM_ERR_INVALID_ARG" in str(err.value)
