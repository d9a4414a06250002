"""Mamba-2 SSD forward on the GPU (through the C ABI) against the f64 SSD
oracle: ragged last chunks, one and several groups, both state sizes, an
initial state and the final state, the limit on delta, a single step, the
full Mamba-2-1.3B shape on sampled heads, and bit-identical repeated calls.
Tolerance: the bf16 I/O bound, normwise max relative error <= 2e-2."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, np64, rel_err
from selective_state_space_s6_gb300 import inputs, s6

pytestmark = pytest.mark.gpu

KEYS = ("x", "dt_raw", "dt_bias", "A_log", "Bm", "Cm", "Dp")


def _dev(x):
    return {k: (v.cuda() if v is not None else None) for k, v in x.items()}


SHAPES = [
    # B, L, H, P, G, N
    (2, 200, 4, 64, 2, 64),    # ragged last chunk, two groups
    (1, 130, 3, 64, 1, 128),
    (2, 64, 2, 64, 1, 128),    # exactly one chunk
    (1, 1, 2, 64, 1, 64),      # a single step
    (3, 300, 6, 64, 3, 128),   # three groups of two heads
    (2, 200, 4, 128, 2, 64),   # headdim 128: two sub-heads per head
    (1, 130, 3, 192, 1, 128),  # headdim 192
    (2, 100, 2, 256, 1, 64),   # headdim 256
    (2, 200, 4, 32, 2, 64),    # headdim 32: run as 64 with the last 32 columns zero
    (1, 130, 3, 32, 1, 128),
]


@pytest.mark.parametrize("B,L,H,P,G,N", SHAPES)
@pytest.mark.parametrize("with_h0", [True, False])
def test_ssd_parity(B, L, H, P, G, N, with_h0):
    x = inputs.make_ssd_inputs(B, L, H, P, G, N, "bf16", seed=B + L + N, h0_std=0.5 if with_h0 else None)
    xd = _dev(x)
    y, h_last = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"])
    s6.check_device_status()
    ry, rh = oracle.ssd_fwd(*[x[k] for k in KEYS], x["h0"])
    assert rel_err(np64(y), ry) <= TOL["bf16"]
    assert rel_err(np64(h_last), rh) <= TOL["bf16"]


def test_ssd_dt_limit():
    x = inputs.make_ssd_inputs(2, 150, 4, 64, 1, 128, "bf16", seed=5, h0_std=0.5)
    sp = torch.nn.functional.softplus(x["dt_raw"].double() + x["dt_bias"].double())
    lim = (float(np.float32(torch.quantile(sp.flatten()[::7].float(), 0.25))),
           float(np.float32(torch.quantile(sp.flatten()[::7].float(), 0.75))))
    xd = _dev(x)
    y, h_last = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"], dt_limit=lim)
    s6.check_device_status()
    ry, rh = oracle.ssd_fwd(*[x[k] for k in KEYS], x["h0"], dt_limit=lim)
    ny, _ = oracle.ssd_fwd(*[x[k] for k in KEYS], x["h0"])
    assert rel_err(ry, ny) > 0.05  # the limit changes the answer
    assert rel_err(np64(y), ry) <= TOL["bf16"]
    assert rel_err(np64(h_last), rh) <= TOL["bf16"]


@pytest.mark.parametrize("N", [64, 128])
def test_ssd_steep_and_mixed_decays(N):
    """Heads whose 8-step decay runs past e^64 (the readout then takes the
    exact per-element exponentials) beside heads near that edge (chunks of
    either kind) and mild ones, in one launch."""
    x = inputs.make_ssd_inputs(2, 260, 6, 64, 2, N, "bf16", seed=31, h0_std=0.5)
    sp_inv = lambda v: float(np.log(np.expm1(v)))  # noqa: E731
    x["dt_bias"] = torch.tensor([sp_inv(3.0), sp_inv(1.0), sp_inv(0.05), sp_inv(6.0), sp_inv(0.9), sp_inv(0.01)],
                                dtype=torch.float32)
    x["A_log"] = torch.log(torch.tensor([16.0, 8.0, 4.0, 2.0, 9.0, 1.0], dtype=torch.float32))
    xd = _dev(x)
    y, h_last = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"])
    s6.check_device_status()
    ry, rh = oracle.ssd_fwd(*[x[k] for k in KEYS], x["h0"])
    for h in range(6):
        assert rel_err(np64(y)[:, :, h], ry[:, :, h]) <= TOL["bf16"], h
    assert rel_err(np64(h_last), rh) <= TOL["bf16"]


def test_ssd_full_shape_sampled_heads():
    w = inputs.SSD_WORKLOADS["mamba2_1p3b"]
    x = inputs.make_ssd_inputs(w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, w.act, seed=0)
    xd = _dev(x)
    y, h_last = s6.ssd_fwd(*[xd[k] for k in KEYS], None)
    s6.check_device_status()
    for b, h in ((0, 0), (1, 33), (3, 63)):
        g = h // (w.nheads // w.ngroups)
        sub = {"x": x["x"][b:b + 1, :, h:h + 1], "dt_raw": x["dt_raw"][b:b + 1, :, h:h + 1],
               "dt_bias": x["dt_bias"][h:h + 1], "A_log": x["A_log"][h:h + 1],
               "Bm": x["Bm"][b:b + 1, :, g:g + 1], "Cm": x["Cm"][b:b + 1, :, g:g + 1], "Dp": x["Dp"][h:h + 1]}
        ry, rh = oracle.ssd_fwd(*[sub[k] for k in KEYS])
        assert rel_err(np64(y[b:b + 1, :, h:h + 1]), ry) <= TOL["bf16"], (b, h)
        assert rel_err(np64(h_last[b:b + 1, h:h + 1]), rh) <= TOL["bf16"], (b, h)


def test_ssd_deterministic():
    x = _dev(inputs.make_ssd_inputs(2, 500, 8, 64, 2, 128, "bf16", seed=7, h0_std=0.5))
    y0, h0 = s6.ssd_fwd(*[x[k] for k in KEYS], x["h0"])
    for _ in range(3):
        y1, h1 = s6.ssd_fwd(*[x[k] for k in KEYS], x["h0"])
        assert torch.equal(y0, y1) and torch.equal(h0, h1)


@pytest.mark.parametrize("B,L,H,G,N", [(1, 1000, 8, 2, 128), (2, 777, 4, 1, 64), (1, 256, 2, 1, 128)])
def test_ssd_split_sequences_match_whole(B, L, H, G, N):
    """With fewer sequences than SMs and h_last requested, each sequence is cut
    in two (a state-only pass to the cut, then both halves at once): y equals
    the uncut walk (no h_last asked) bit for bit, h_last matches the oracle."""
    x = inputs.make_ssd_inputs(B, L, H, 64, G, N, "bf16", seed=B + L + H, h0_std=0.5)
    xd = _dev(x)
    y_split, h_split = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"])
    y_whole, none = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"], want_h_last=False)
    s6.check_device_status()
    assert none is None
    assert torch.equal(y_split, y_whole)
    ry, rh = oracle.ssd_fwd(*[x[k] for k in KEYS], x["h0"])
    assert rel_err(np64(y_split), ry) <= TOL["bf16"]
    assert rel_err(np64(h_split), rh) <= TOL["bf16"]


def test_ssd_wide_heads_split_match_whole():
    """Headdim 128 on few sequences (16 sub-head sequences: cut in two): y
    equals the uncut walk bit for bit and matches the oracle, with h_last."""
    x = inputs.make_ssd_inputs(1, 1000, 8, 128, 2, 128, "bf16", seed=77, h0_std=0.5)
    xd = _dev(x)
    y_split, h_split = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"])
    y_whole, _ = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"], want_h_last=False)
    s6.check_device_status()
    assert torch.equal(y_split, y_whole)
    ry, rh = oracle.ssd_fwd(*[x[k] for k in KEYS], x["h0"])
    assert rel_err(np64(y_split), ry) <= TOL["bf16"]
    assert rel_err(np64(h_split), rh) <= TOL["bf16"]


def test_ssd_state_in_place():
    """h0 and h_last as one buffer (the state updated in place), on a shape
    that would otherwise be cut in two: same y and final state as separate
    buffers."""
    x = _dev(inputs.make_ssd_inputs(1, 1000, 8, 64, 2, 128, "bf16", seed=41, h0_std=0.5))
    y_ref, h_ref = s6.ssd_fwd(*[x[k] for k in KEYS], x["h0"])
    state = x["h0"].clone()
    y_in, h_in = s6.ssd_fwd(*[x[k] for k in KEYS], state, h_last=state)
    s6.check_device_status()
    assert h_in.data_ptr() == state.data_ptr()
    assert torch.equal(y_in, y_ref)
    assert torch.equal(state, h_ref)


def test_ssd_empty_sequence_keeps_the_state():
    x = _dev(inputs.make_ssd_inputs(2, 0, 2, 64, 1, 64, "bf16", seed=1, h0_std=0.5))
    y, h_last = s6.ssd_fwd(*[x[k] for k in KEYS], x["h0"])
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.equal(h_last, x["h0"])


def _sweep(n=8, seed=321):
    r = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B = int(r.integers(1, 4))
        L = int(r.integers(1, 300))
        G = int(r.integers(1, 4))
        H = G * int(r.integers(1, 4))
        N = int(r.choice([64, 128]))
        h0 = bool(r.integers(0, 2))
        lim = bool(r.integers(0, 2))
        out.append((B, L, H, G, N, h0, lim))
    return out


@pytest.mark.parametrize("B,L,H,G,N,with_h0,limited", _sweep())
def test_ssd_random_shape_sweep(B, L, H, G, N, with_h0, limited):
    """Seeded random shapes (lengths from one step to several ragged chunks,
    groups, both state sizes, with and without h0 and a limit on delta)."""
    x = inputs.make_ssd_inputs(B, L, H, 64, G, N, "bf16", seed=B * 7 + L, h0_std=0.5 if with_h0 else None)
    lim = (0.01, 0.05) if limited else None
    xd = _dev(x)
    y, h_last = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"], dt_limit=lim)
    s6.check_device_status()
    ry, rh = oracle.ssd_fwd(*[x[k] for k in KEYS], x["h0"], dt_limit=lim)
    assert rel_err(np64(y), ry) <= TOL["bf16"]
    assert rel_err(np64(h_last), rh) <= TOL["bf16"]


def _wide_sweep(n=6, seed=654):
    r = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B = int(r.integers(1, 3))
        L = int(r.integers(1, 300))
        G = int(r.integers(1, 3))
        H = G * int(r.integers(1, 3))
        N = int(r.choice([64, 128]))
        P = int(r.choice([128, 192, 256]))
        out.append((B, L, H, G, N, P, bool(r.integers(0, 2)), bool(r.integers(0, 2))))
    return out


@pytest.mark.parametrize("B,L,H,G,N,P,with_h0,limited", _wide_sweep())
def test_ssd_wide_random_shape_sweep(B, L, H, G, N, P, with_h0, limited):
    """Seeded random shapes with heads of 128-256 columns."""
    x = inputs.make_ssd_inputs(B, L, H, P, G, N, "bf16", seed=B * 5 + L + P, h0_std=0.5 if with_h0 else None)
    lim = (0.01, 0.05) if limited else None
    xd = _dev(x)
    y, h_last = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"], dt_limit=lim)
    s6.check_device_status()
    ry, rh = oracle.ssd_fwd(*[x[k] for k in KEYS], x["h0"], dt_limit=lim)
    assert rel_err(np64(y), ry) <= TOL["bf16"]
    assert rel_err(np64(h_last), rh) <= TOL["bf16"]
