"""Causal depthwise conv1d + SiLU on the GPU (through the C ABI) against the
f64 conv1d oracle: forward with and without an initial state, the final
state, backward with every gradient, the single step against the multi-step
forward (bit for bit), the state hand-over between two calls, bit-identical
gradients over repeated calls, and the empty and ragged edge cases."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, np64, rel_err
from selective_state_space_s6_gb300 import s6

pytestmark = pytest.mark.gpu


def _case(B, L, D, K, act, seed, state=True):
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if act == "bf16" else torch.float32
    x = torch.randn(B, L, D, generator=g).to(dt)
    w = (torch.randn(D, K, generator=g) * 0.5).float()
    bias = (torch.randn(D, generator=g) * 0.2).float()
    s0 = torch.randn(B, D, K - 1, generator=g).to(dt) if state else None
    dout = torch.randn(B, L, D, generator=g).to(dt)
    return x, w, bias, s0, dout


def _dev(*ts):
    return [None if t is None else t.cuda() for t in ts]


# (B, L, D, K, act, kernel path of both directions)
SHAPES = [
    (2, 100, 64, 4, "f32", "tile"), (2, 100, 64, 4, "bf16", "tile"),
    (3, 67, 37, 4, "f32", "scalar"), (1, 130, 21, 3, "bf16", "scalar"),  # odd channel counts
    (2, 100, 12, 4, "bf16", "vector"),        # rows of 24 bytes: no tensor map
    (2, 2, 16, 4, "f32", "tile"),             # shorter than the window
    (3, 1, 8, 4, "bf16", "tile"),             # a single step
    (1, 200, 32, 1, "f32", "tile"), (2, 150, 24, 8, "bf16", "tile"),  # width 1 and the widest
    (2, 129, 256, 4, "bf16", "tile"),         # ragged last tile of 64 steps
    (2, 300, 200, 5, "f32", "tile"),          # ragged channel tile (128 + 72)
    (1, 70, 136, 8, "bf16", "tile"),          # channel tile of 8, widest window
]


@pytest.mark.parametrize("B,L,D,K,act,path", SHAPES)
@pytest.mark.parametrize("state", [True, False])
def test_conv1d_fwd_bwd_parity(B, L, D, K, act, path, state):
    x, w, bias, s0, dout = _case(B, L, D, K, act, seed=B + L + K, state=state)
    xd, wd, bd, sd, dd = _dev(x, w, bias, s0, dout)
    assert s6.conv1d_path(xd, wd) == path
    assert s6.conv1d_path(xd, wd, dout=dd, y=torch.empty_like(dd)) == path
    out, s_last = s6.conv1d_fwd(xd, wd, bd, sd)
    g = s6.conv1d_bwd(xd, wd, bd, sd, dd)
    torch.cuda.synchronize()
    ref_out, ref_s = oracle.conv1d_fwd(x, w, bias, s0)
    ref = oracle.conv1d_bwd(x, w, bias, s0, dout)
    tol = TOL[act]
    assert rel_err(np64(out), ref_out) <= tol
    if K > 1:
        assert np.array_equal(np64(s_last), ref_s)  # copies of inputs: exact
    for k in ("dx", "dw", "dbias"):
        assert rel_err(np64(g[k]), ref[k]) <= tol, k
    if K > 1:
        assert rel_err(np64(g["dstate0"]), ref["dstate0"]) <= tol


def test_conv1d_step_chain_equals_forward_bitwise():
    B, L, D, K = 3, 40, 48, 4
    for act in ("f32", "bf16"):
        x, w, bias, s0, _ = _case(B, L, D, K, act, seed=5)
        xd, wd, bd, sd = _dev(x, w, bias, s0)
        out, s_last = s6.conv1d_fwd(xd, wd, bd, sd)
        st = sd.clone()
        outs = [s6.conv1d_step(xd[:, t].contiguous(), wd, bd, st) for t in range(L)]
        assert torch.equal(torch.stack(outs, dim=1), out)
        assert torch.equal(st, s_last)


def test_conv1d_state_handover_bitwise():
    x, w, bias, s0, _ = _case(2, 300, 64, 4, "bf16", seed=6)
    xd, wd, bd, sd = _dev(x, w, bias, s0)
    out, s_last = s6.conv1d_fwd(xd, wd, bd, sd)
    o1, s_mid = s6.conv1d_fwd(xd[:, :137].contiguous(), wd, bd, sd)
    o2, s_end = s6.conv1d_fwd(xd[:, 137:].contiguous(), wd, bd, s_mid)
    assert torch.equal(torch.cat([o1, o2], dim=1), out)
    assert torch.equal(s_end, s_last)


def test_conv1d_backward_deterministic():
    x, w, bias, s0, dout = _case(4, 700, 512, 4, "bf16", seed=7)
    xd, wd, bd, sd, dd = _dev(x, w, bias, s0, dout)
    first = s6.conv1d_bwd(xd, wd, bd, sd, dd)
    for _ in range(4):
        again = s6.conv1d_bwd(xd, wd, bd, sd, dd)
        for k in first:
            assert torch.equal(first[k], again[k]), k


def test_conv1d_empty():
    w = torch.randn(8, 4).cuda()
    bias = torch.randn(8).cuda()
    x = torch.empty(2, 0, 8).cuda()
    s0 = torch.randn(2, 8, 3).cuda()
    out, s_last = s6.conv1d_fwd(x, w, bias, s0)
    assert out.shape == (2, 0, 8) and torch.equal(s_last, s0)
    g = s6.conv1d_bwd(x, w, bias, s0, torch.empty_like(x))
    torch.cuda.synchronize()
    assert torch.count_nonzero(g["dw"]) == 0 and torch.count_nonzero(g["dbias"]) == 0
    assert torch.count_nonzero(g["dstate0"]) == 0


def _offset_copy(t, elems):
    """A copy of ``t`` whose data starts ``elems`` elements into a fresh buffer
    (to steer the kernel choice by alignment)."""
    buf = torch.empty(t.numel() + elems, dtype=t.dtype, device=t.device)
    v = buf[elems:].view(t.shape)
    v.copy_(t)
    return v


def test_conv1d_paths_agree():
    """The tile, vector and scalar kernels on the same bf16 problem, steered
    by the alignment of x, dout, out and dx: forward outputs and dx agree bit
    for bit (same arithmetic per element); dw and dbias, summed in other
    orders, agree to rounding."""
    B, L, D, K = 2, 333, 192, 4
    x, w, bias, s0, dout = _case(B, L, D, K, "bf16", seed=8)
    xd, wd, bd, sd, dd = _dev(x, w, bias, s0, dout)
    res = {}
    for off, path in ((0, "tile"), (4, "vector"), (1, "scalar")):
        xo, do = _offset_copy(xd, off), _offset_copy(dd, off)
        out = _offset_copy(torch.empty_like(xd), off)
        assert s6.conv1d_path(xo, wd, y=out) == path
        s6.conv1d_fwd(xo, wd, bd, sd, out=out)
        dx = _offset_copy(torch.empty_like(xd), off)
        assert s6.conv1d_path(xo, wd, dout=do, y=dx) == path
        g = s6.conv1d_bwd(xo, wd, bd, sd, do, dx=dx)
        res[path] = (out.clone(), g)
    torch.cuda.synchronize()
    ref_out, ref_g = res["tile"]
    for path in ("vector", "scalar"):
        out, g = res[path]
        assert torch.equal(out, ref_out), path
        assert torch.equal(g["dx"], ref_g["dx"]), path
        for k in ("dw", "dbias", "dstate0"):
            assert rel_err(np64(g[k]), np64(ref_g[k])) <= 1e-5, (path, k)


def _sweep_shapes(n=10, seed=123):
    r = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B = int(r.integers(1, 4))
        L = int(r.integers(1, 400))
        D = int(r.choice([8, 24, 40, 64, 100, 136, 264]))
        K = int(r.integers(1, 9))
        act = str(r.choice(["f32", "bf16"]))
        state = bool(r.integers(0, 2))
        out.append((B, L, D, K, act, state))
    return out


@pytest.mark.parametrize("B,L,D,K,act,state", _sweep_shapes())
def test_conv1d_random_shape_sweep(B, L, D, K, act, state):
    """Seeded random shapes over every path, width and edge (L < K, ragged
    tiles and channel tiles), forward and backward against the oracle."""
    x, w, bias, s0, dout = _case(B, L, D, K, act, seed=B * 31 + L + K, state=state)
    xd, wd, bd, sd, dd = _dev(x, w, bias, s0, dout)
    out, s_last = s6.conv1d_fwd(xd, wd, bd, sd)
    g = s6.conv1d_bwd(xd, wd, bd, sd, dd)
    torch.cuda.synchronize()
    ref_out, ref_s = oracle.conv1d_fwd(x, w, bias, s0)
    ref = oracle.conv1d_bwd(x, w, bias, s0, dout)
    tol = TOL[act]
    assert rel_err(np64(out), ref_out) <= tol
    if K > 1:
        assert np.array_equal(np64(s_last), ref_s)
    for k in ("dx", "dw", "dbias"):
        assert rel_err(np64(g[k]), ref[k]) <= tol, k
