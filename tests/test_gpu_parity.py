"""Parity of the CUDA path (through the C ABI) with the f64 oracle.

Small shapes are compared element by element on every output; they span
several channel tiles and chunks with ragged tails, every state count 1..16
(padded lanes), with and without the gate, initial state and final-state
gradient.  The full-size workloads are compared element by element on every
output too, in the launch configuration the benchmark times.
"""
import hashlib

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (ARGS, GRAD_KEYS, TOL, act_of, compare_all, gpu_fwd_bwd, np64,
                         oracle_fwd_bwd, rel_err, to_dev)
from selective_state_space_s6_gb300 import inputs, s6

pytestmark = pytest.mark.gpu


def _inputs(B, L, D, N, act, seed=0, z=True, h0=True, dh=True, **kw):
    return inputs.make_inputs(B, L, D, N, act, seed=seed, with_z=z,
                              h0_std=0.5 if h0 else None, with_dh_last=dh, **kw)


SMALL = [
    # B, L, D, N, act
    (1, 64, 16, 4, "f32"),     # the tiny workload's shape
    (2, 1, 3, 1, "f32"),       # single step, single state
    (1, 65, 17, 3, "f32"),     # ragged chunk and tile (65 = 2*32 + 1), odd N
    (3, 130, 70, 16, "f32"),   # two tiles, three chunks
    (2, 200, 65, 5, "bf16"),
    (1, 64, 64, 16, "bf16"),
    (2, 129, 128, 8, "f32"),
    (1, 300, 33, 2, "bf16"),
    (1, 77, 130, 16, "bf16"),
    # shapes on the TMA path (N*e and D*e multiples of 16 bytes) with ragged tails
    (2, 100, 72, 16, "bf16"),   # ragged 64-channel tile, L not a multiple of 32 or 64
    (1, 33, 8, 8, "bf16"),      # a tile that is mostly out of bounds
    (3, 95, 136, 16, "f32"),
    (1, 1, 64, 16, "bf16"),     # one step
    (2, 31, 24, 4, "f32"),
    (2, 160, 64, 8, "f32"),
    # long and narrow: the forward splits time into segments (chunked parallel scan)
    (1, 1100, 64, 16, "f32"),   # 2 segments, ragged last one
    (1, 4096, 32, 16, "bf16"),  # 8 segments of 512 steps
    (2, 3000, 100, 4, "f32"),   # 128 channels per tile, 5 segments
    (1, 2500, 72, 8, "bf16"),
]


@pytest.mark.parametrize("B,L,D,N,act", SMALL)
@pytest.mark.parametrize("variant", ["full", "nogate_noh0"])
def test_small_parity(B, L, D, N, act, variant):
    full = variant == "full"
    x = _inputs(B, L, D, N, act, seed=B * 1000 + L + D + N, z=full, h0=full, dh=full)
    gpu = gpu_fwd_bwd(to_dev(x), dh_last=x["dh_last"].cuda() if full else None)
    ref = oracle_fwd_bwd(x, dh_last=x["dh_last"])
    errs = compare_all(gpu, ref, TOL[act])
    assert errs


def test_tiny_workload_every_output_and_chunk_states():
    x = inputs.make_workload("tiny")
    gpu = gpu_fwd_bwd(to_dev(x))
    ref = oracle_fwd_bwd(x)
    compare_all(gpu, ref, TOL["f32"])
    # chunk state c = state before step c*CHUNK_LEN = h_last of the first c*CHUNK_LEN steps
    cl = s6.CHUNK_LEN
    x2 = _inputs(2, 200, 24, 16, "f32", seed=5)
    g2 = gpu_fwd_bwd(to_dev(x2), want_bwd=False)
    cs = np64(g2["chunk_states"])
    nc = -(-200 // cl)
    assert cs.shape == (2, nc, 24, 16)
    assert np.array_equal(cs[:, 0], x2["h0"].double().numpy())
    for c in range(1, nc):
        sub = {k: (v[:, : c * cl].contiguous() if k in ("u", "delta_raw", "z", "Bm", "Cm") else v)
               for k, v in x2.items()}
        _, h_ref = oracle.fwd(*[sub[k] for k in ARGS], sub["h0"])
        assert rel_err(cs[:, c], h_ref) <= TOL["f32"]


def test_nosave_matches_save():
    x = to_dev(_inputs(2, 150, 70, 16, "bf16", seed=3))
    o1, h1, _ = s6.ssm_scan_fwd(*[x[k] for k in ARGS], x["h0"])
    o2, h2 = s6.ssm_scan_fwd_nosave(*[x[k] for k in ARGS], x["h0"])
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


STEP_SHAPES = [
    # B, L, D, N, act, gate
    (3, 40, 70, 16, "f32", True),    # D*4 not a multiple of 16: generic scan and step
    (3, 40, 70, 16, "bf16", True),
    (2, 45, 64, 16, "f32", True),    # TMA scan and the dedicated step kernel
    (3, 33, 200, 16, "bf16", True),  # ragged channel tile
    (2, 37, 32, 8, "f32", False),    # two lanes per channel, no gate
    (2, 30, 64, 8, "bf16", True),
    (3, 29, 24, 4, "f32", True),     # one lane per channel
]


@pytest.mark.parametrize("B,L,D,N,act,gate", STEP_SHAPES)
def test_step_chain_equals_scan(B, L, D, N, act, gate):
    x = _inputs(B, L, D, N, act, seed=11, z=gate)
    xd = to_dev(x)
    out_scan, h_scan, _ = s6.ssm_scan_fwd(*[xd[k] for k in ARGS], xd["h0"])
    h = xd["h0"].clone()
    outs = []
    for t in range(L):
        sl = {k: (xd[k][:, t].contiguous() if xd[k] is not None else None)
              for k in ("u", "delta_raw", "z", "Bm", "Cm")}
        outs.append(s6.ssm_step(sl["u"], sl["delta_raw"], sl["z"], sl["Bm"], sl["Cm"],
                                xd["A_log"], xd["Dp"], xd["delta_bias"], h))
    out_step = torch.stack(outs, dim=1)
    # same per-step arithmetic in registers vs. through memory: bit-identical
    assert torch.equal(out_step, out_scan)
    assert torch.equal(h, h_scan)
    ref_out, ref_h = oracle.fwd(*[x[k] for k in ARGS], x["h0"])
    assert rel_err(np64(out_step), ref_out) <= TOL[act]
    assert rel_err(np64(h), ref_h) <= TOL[act]


def _digest(tensors):
    m = hashlib.sha256()
    for t in tensors:
        if t is not None:
            m.update(t.detach().contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return m.hexdigest()


@pytest.mark.parametrize("shape", [(1, 64, 16, 4, "f32"), (3, 700, 200, 16, "bf16")])
def test_bitwise_deterministic_10_runs(shape):
    x = to_dev(_inputs(*shape, seed=21))
    digests = set()
    for _ in range(10):
        r = gpu_fwd_bwd(x, dh_last=x["dh_last"])
        digests.add(_digest([r["out"], r["h_last"], r["chunk_states"]] + [r[k] for k in GRAD_KEYS]))
    assert len(digests) == 1


@pytest.mark.parametrize("name", ["mamba130m", "mamba1p4b", "long"])
def test_bitwise_deterministic_10_runs_full_size(name):
    """Ten forward + backward runs of a full-size workload give identical
    bytes in every output (compared on the device against the first run)."""
    xd = to_dev(inputs.make_workload(name))
    first = gpu_fwd_bwd(xd)
    keep = {k: v.clone() for k, v in first.items() if v is not None}
    for _ in range(9):
        r = gpu_fwd_bwd(xd)
        for k, v in keep.items():
            assert torch.equal(r[k], v), k


def test_empty_inputs():
    # L = 0: no steps; h_last = h0, parameter gradients 0, dh0 = dh_last
    x = to_dev(_inputs(2, 0, 5, 3, "f32", seed=1))
    r = gpu_fwd_bwd(x, dh_last=x["dh_last"])
    assert r["out"].numel() == 0 and r["chunk_states"].numel() == 0
    assert torch.equal(r["h_last"], x["h0"])
    assert torch.equal(r["dh0"], x["dh_last"])
    for k in ("dA_log", "dD", "d_delta_bias"):
        assert torch.count_nonzero(r[k]) == 0
    # B = 0: parameter gradients 0
    x = to_dev(_inputs(0, 10, 5, 3, "bf16", seed=1))
    r = gpu_fwd_bwd(x)
    for k in ("dA_log", "dD", "d_delta_bias"):
        assert torch.count_nonzero(r[k]) == 0
    # D = 0: nothing to do, no error
    x = to_dev(_inputs(2, 10, 0, 3, "f32", seed=1))
    gpu_fwd_bwd(x)
    torch.cuda.synchronize()


def test_extreme_decay_and_skip():
    """Large |A| (state resets every step) and delta -> 0 (skip path only)."""
    x = _inputs(2, 100, 70, 16, "f32", seed=8)
    x["A_log"] = torch.full_like(x["A_log"], 60.0)
    gpu = gpu_fwd_bwd(to_dev(x), dh_last=x["dh_last"].cuda())
    ref = oracle_fwd_bwd(x, dh_last=x["dh_last"])
    compare_all(gpu, ref, TOL["f32"])
    x = _inputs(2, 100, 70, 16, "f32", seed=9)
    x["delta_raw"] = torch.full_like(x["delta_raw"], -120.0)  # softplus underflows in f32
    gpu = gpu_fwd_bwd(to_dev(x), dh_last=x["dh_last"].cuda())
    ref = oracle_fwd_bwd(x, dh_last=x["dh_last"])
    compare_all(gpu, ref, TOL["f32"], keys=("out", "h_last", "du", "dz", "dCm", "dD", "dh0"))
    # the rest scale with delta ~ e^-120 in the oracle and must be (close to) zero here
    for k in ("d_delta_raw", "dBm", "dA_log", "d_delta_bias"):
        assert float(torch.max(torch.abs(gpu[k]))) <= 1e-30, k


# ------------------------------------------------------------------ full-size workloads

BLD = ("u", "delta_raw", "z", "dout")
# dh0 on the long workload: the f32 floor there is 1.46e-5 (see below)
LONG_DH0_TOL = 1e-4


def _batch_rows(x, b0, b1):
    """The sub-problem on batch rows b0..b1-1 (per-batch inputs sliced, parameters kept)."""
    y = {}
    for k, v in x.items():
        if v is None or k in ("A_log", "Dp", "delta_bias"):
            y[k] = v
        else:
            y[k] = v[b0:b1].contiguous()
    return y


@pytest.mark.parametrize("name", ["mamba130m", "mamba1p4b", "long"])
def test_full_size_every_output(name):
    """The full-size workloads, in the launch configuration the benchmark
    times: every element of every output and gradient (out, h_last, du,
    d_delta_raw, dz, dBm, dCm, dA_log, dDp, d_delta_bias, dh0) against the
    oracle on the whole problem, at the workload's tolerance."""
    x = inputs.make_workload(name)
    act = inputs.WORKLOADS[name].act
    xd = to_dev(x)
    gpu = gpu_fwd_bwd(xd, dh_last=xd["dh_last"])
    gpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in gpu.items()}
    del xd
    torch.cuda.empty_cache()
    ref = oracle_fwd_bwd(x, dh_last=x["dh_last"])
    keys = ("out", "h_last", "du", "d_delta_raw", "dz", "dBm", "dCm", "dA_log", "dD", "d_delta_bias", "dh0")
    if name == "long":
        # dh0 of the 65536-step sequence: the adjoint of the slowest state
        # (delta ~ 1.2e-4, A = -1) sums ~8000 steps, and f32 itself cannot hold
        # 1e-5 there -- the plain sequential f32 recurrence (one rounding per
        # operation) is 1.46e-5 from the oracle on this output.  Its bound is
        # LONG_DH0_TOL; every other output keeps the f32 tolerance.
        errs = compare_all(gpu, ref, TOL[act], keys=keys[:-1])
        errs.update(compare_all(gpu, ref, LONG_DH0_TOL, keys=("dh0",)))
    else:
        errs = compare_all(gpu, ref, TOL[act], keys=keys)
    assert set(errs) >= set(keys), errs


def test_decode_1000_chained_steps():
    """1000 chained decode steps (B=256, D=1536, N=16, f32) equal the scan over
    the same tokens bit for bit, and every output and the final state match
    the oracle's scan (compared in slices of 32 batch rows)."""
    w = inputs.WORKLOADS["decode"]
    x = inputs.make_workload("decode", with_dout=False)
    xd = to_dev(x)
    h = xd["h0"].clone()
    out_steps = torch.empty_like(xd["u"])
    for t in range(w.seqlen):
        sl = {k: xd[k][:, t].contiguous() for k in ("u", "delta_raw", "z", "Bm", "Cm")}
        out_steps[:, t] = s6.ssm_step(sl["u"], sl["delta_raw"], sl["z"], sl["Bm"], sl["Cm"],
                                      xd["A_log"], xd["Dp"], xd["delta_bias"], h)
    out_scan, h_scan, _ = s6.ssm_scan_fwd(*[xd[k] for k in ARGS], xd["h0"], save=False)
    assert torch.equal(out_steps, out_scan)
    assert torch.equal(h, h_scan)
    out_cpu, h_cpu = out_steps.cpu(), h.cpu()
    del xd, out_steps, out_scan, h_scan
    torch.cuda.empty_cache()
    diff_o = diff_h = scale_o = scale_h = 0.0
    for b0 in range(0, w.batch, 32):
        xs = _batch_rows(x, b0, min(w.batch, b0 + 32))
        ref_out, ref_h = oracle.fwd(*[xs[k] for k in ARGS], xs["h0"])
        diff_o = max(diff_o, float(np.max(np.abs(np64(out_cpu[b0:b0 + 32]) - ref_out))))
        diff_h = max(diff_h, float(np.max(np.abs(np64(h_cpu[b0:b0 + 32]) - ref_h))))
        scale_o = max(scale_o, float(np.max(np.abs(ref_out))))
        scale_h = max(scale_h, float(np.max(np.abs(ref_h))))
    assert diff_o / scale_o <= TOL["f32"], diff_o / scale_o
    assert diff_h / scale_h <= TOL["f32"], diff_h / scale_h


@pytest.mark.parametrize("B,L,D,N,act", [(4, 256, 5120, 16, "bf16"), (3, 192, 8192, 16, "f32")])
def test_handover_mode(B, L, D, N, act):
    """Shapes whose backward cuts every (batch, channel tile) sequence at most
    once, with ranges longer than a sequence: the carry is handed from the CTA
    walking a sequence's last piece to the one walking its first piece.  Every
    output against the oracle, and bit-identical over two runs."""
    assert s6.plan_segments(B, L, D, N, s6.SSM_BF16 if act == "bf16" else s6.SSM_F32)[1] == 1
    x = _inputs(B, L, D, N, act, seed=21)
    xd = to_dev(x)
    got = gpu_fwd_bwd(xd, dh_last=xd["dh_last"])
    again = gpu_fwd_bwd(xd, dh_last=xd["dh_last"])
    for k in GRAD_KEYS:
        if got.get(k) is not None:
            assert torch.equal(got[k], again[k]), k
    ref = oracle_fwd_bwd(x, dh_last=x["dh_last"])
    compare_all(got, ref, TOL[act])


def _sweep_shapes(n=14, seed=1234):
    """Seeded random shapes over the plan's regimes: dstate 4/8/16 (TMA path)
    and others (generic path), ragged channel tiles and chunks, both dtypes."""
    rng = np.random.default_rng(seed)
    shapes = []
    for _ in range(n):
        act = "bf16" if rng.random() < 0.5 else "f32"
        N = int(rng.choice([4, 8, 16, 16, 16, 6])) if act == "f32" else int(rng.choice([8, 16, 16]))
        B = int(rng.integers(1, 5))
        L = int(rng.integers(1, 700))
        D = int(rng.integers(1, 40)) * 8
        shapes.append((B, L, D, N, act))
    return shapes


@pytest.mark.parametrize("B,L,D,N,act", _sweep_shapes())
def test_random_shape_sweep(B, L, D, N, act):
    x = _inputs(B, L, D, N, act, seed=B * 7 + L)
    gpu = gpu_fwd_bwd(to_dev(x), dh_last=to_dev(x)["dh_last"])
    ref = oracle_fwd_bwd(x, dh_last=x["dh_last"])
    compare_all(gpu, ref, TOL[act])


@pytest.mark.parametrize("B,L,D,N,act", [(5, 192, 3072, 16, "f32"), (4, 160, 4096, 16, "bf16")])
def test_forward_stream_mode(B, L, D, N, act):
    """Shapes whose forward runs in stream mode (3 CTAs per SM over equal
    ranges of chunks, the state of a cut sequence handed from CTA to CTA):
    outputs, final state and chunk states against the oracle."""
    a = s6.SSM_BF16 if act == "bf16" else s6.SSM_F32
    assert s6.plan_segments(B, L, D, N, a)[0] == 1 and s6.fwd_workspace_bytes(B, L, D, N, a) > 0
    x = _inputs(B, L, D, N, act, seed=31)
    xd = to_dev(x)
    got = gpu_fwd_bwd(xd, dh_last=xd["dh_last"])
    ref = oracle_fwd_bwd(x, dh_last=x["dh_last"])
    compare_all(got, ref, TOL[act])
    cl = s6.CHUNK_LEN
    cs = np64(got["chunk_states"])
    for c in (1, (L - 1) // cl):
        sub = {k: (v[:, : c * cl].contiguous() if k in ("u", "delta_raw", "z", "Bm", "Cm") else v)
               for k, v in x.items()}
        _, h_ref = oracle.fwd(*[sub[k] for k in ARGS], sub["h0"])
        assert rel_err(cs[:, c], h_ref) <= TOL[act]


@pytest.mark.parametrize("B,L,D,N,act", [(2, 300, 72, 16, "f32"), (3, 700, 200, 8, "f32"),
                                         (2, 500, 128, 16, "bf16"), (1, 4096, 256, 16, "bf16")])
def test_gpu_gradients_internally_consistent(B, L, D, N, act):
    """The identities d_delta_bias = sum_{b,t} d_delta_raw and
    dD = sum_{b,t} dy * u (dy = dout * silu(z)) hold for the GPU's own
    outputs: d_delta_raw re-summed from the returned tensor, dy formed in f64
    from the inputs (the sums that produce d_delta_bias and dD run on the
    device in a fixed order, separately from the per-step outputs)."""
    x = _inputs(B, L, D, N, act, seed=B * 7 + L + D)
    xd = to_dev(x)
    r = gpu_fwd_bwd(xd, dh_last=xd["dh_last"])
    assert rel_err(np64(r["d_delta_bias"]), np64(r["d_delta_raw"]).sum(axis=(0, 1))) <= TOL[act]
    z, dout, u = np64(xd["z"]), np64(xd["dout"]), np64(xd["u"])
    dy = dout * z / (1.0 + np.exp(-z))
    assert rel_err(np64(r["dD"]), (dy * u).sum(axis=(0, 1))) <= TOL[act]
