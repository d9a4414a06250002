"""Mamba-2 SSD backward on the GPU (through the C ABI) against the f64 SSD
oracle's backward: every gradient (dx, ddt_raw, ddt_bias, dA_log, dBm, dCm,
dDp, dh0) on ragged chunks, one and several groups, both state sizes, with
and without an initial state and a final-state gradient, the limit on delta,
a single step, sequences the forward cuts in two; the state saves of the
forward; bit-identical repeated calls; the full Mamba-2-1.3B shape (per-head
gradients on sampled heads against the oracle over every batch row, the
group sums dBm/dCm through identities that hold at any size).
Tolerance: the bf16 I/O bound, normwise max relative error <= 2e-2."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, np64, rel_err
from selective_state_space_s6_gb300 import inputs, s6

pytestmark = pytest.mark.gpu

KEYS = ("x", "dt_raw", "dt_bias", "A_log", "Bm", "Cm", "Dp")
GRADS = ("dx", "ddt_raw", "ddt_bias", "dA_log", "dBm", "dCm", "dDp", "dh0")


def _dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _problem(B, L, H, G, N, seed, h0=True, dh=True, P=64):
    x = inputs.make_ssd_inputs(B, L, H, P, G, N, "bf16", seed=seed, h0_std=0.5 if h0 else None)
    gen = torch.Generator().manual_seed(seed + 1000)
    x["dy"] = torch.randn((B, L, H, P), generator=gen).to(torch.bfloat16)
    x["dh_last"] = torch.randn((B, H, N, P), generator=gen) if dh else None
    return x


def _gpu(xd, dt_limit=None):
    y, h_last, cs = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"], save=True, dt_limit=dt_limit)
    g = s6.ssd_bwd(*[xd[k] for k in KEYS], cs, xd["dy"], xd["dh_last"], dt_limit=dt_limit)
    s6.check_device_status()
    return y, h_last, cs, g


def _oracle(x, dt_limit=None):
    return oracle.ssd_bwd(*[x[k] for k in KEYS], x["h0"], x["dy"], x["dh_last"], dt_limit=dt_limit)


def _compare(g, ref, tol=TOL["bf16"], keys=GRADS):
    errs = {k: rel_err(np64(g[k]), ref[k]) for k in keys if g.get(k) is not None}
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"errors above {tol}: {bad} (all {errs})"
    return errs


SHAPES = [
    # B, L, H, G, N
    (2, 200, 4, 2, 64),     # ragged last chunk, two groups
    (1, 130, 3, 1, 128),
    (2, 64, 2, 1, 128),     # exactly one chunk
    (1, 1, 2, 1, 64),       # a single step
    (3, 300, 6, 3, 128),    # three groups of two heads
    (1, 1000, 8, 2, 128),   # few sequences: the forward cuts each in two
]


@pytest.mark.parametrize("B,L,H,G,N", SHAPES)
@pytest.mark.parametrize("variant", ["h0_dh", "plain"])
def test_ssd_bwd_parity(B, L, H, G, N, variant):
    full = variant == "h0_dh"
    x = _problem(B, L, H, G, N, seed=B + L + N + H, h0=full, dh=full)
    _, _, _, g = _gpu(_dev(x))
    ref = _oracle(x)
    _compare(g, ref)


def _split_heads(x, P):
    """The problem with each head of P = 64 m columns written as m heads of 64
    (columns split, the head's dt, dt_bias, A_log, Dp repeated)."""
    m = P // 64
    B, L, H, _ = x["x"].shape
    N = x["Bm"].shape[3]
    y = {"Bm": x["Bm"], "Cm": x["Cm"]}
    for k in ("x", "dy"):
        y[k] = x[k].reshape(B, L, H * m, 64).contiguous()
    y["dt_raw"] = x["dt_raw"].repeat_interleave(m, dim=2).contiguous()
    for k in ("dt_bias", "A_log", "Dp"):
        y[k] = x[k].repeat_interleave(m).contiguous()
    for k in ("h0", "dh_last"):
        y[k] = (None if x[k] is None else
                x[k].reshape(B, H, N, m, 64).permute(0, 1, 3, 2, 4).reshape(B, H * m, N, 64).contiguous())
    return y


def _compare_wide(g, x, P, dt_limit=None):
    """Every gradient against the oracle.  The per-head sums (dA_log,
    ddt_bias, dDp) of a head of m sub-heads: the normwise bound (TOL times
    the largest head's magnitude), raised for a head to TOL times the sum of
    the magnitudes of its sub-heads' parts (from the oracle on the split
    problem) -- a head's value is a sum over its columns, which may cancel,
    so its error is bounded by its parts' magnitudes, not by its own."""
    ref = _oracle(x, dt_limit=dt_limit)
    _compare(g, ref, keys=("dx", "ddt_raw", "dBm", "dCm", "dh0"))
    m = P // 64
    parts = _oracle(_split_heads(x, P), dt_limit=dt_limit)
    for k in ("dA_log", "ddt_bias", "dDp"):
        mag = np.abs(parts[k]).reshape(-1, m).sum(axis=1)
        err = np.abs(np64(g[k]) - ref[k])
        bound = TOL["bf16"] * np.maximum(mag, np.abs(ref[k]).max())
        assert np.all(err <= bound + 1e-6), (k, err, bound)
        # the oracle's head is the sum of its parts
        assert np.allclose(parts[k].reshape(-1, m).sum(axis=1), ref[k], rtol=1e-9, atol=1e-9), k


HANDOVER = [
    # B, L, H, G, N, P: more (batch, sub-head) sequences than SMs, so one
    # range of chunks per SM, sequences cut in two and the state gradient
    # handed from the CTA walking a sequence's last piece to the one walking
    # its first
    (2, 200, 80, 2, 64, 64),    # 160 sequences of 4 chunks
    (3, 130, 64, 1, 128, 64),   # 192 of 3, a ragged last chunk
    (1, 300, 160, 4, 128, 64),  # 160 of 5, four groups
    (2, 100, 20, 2, 64, 256),   # headdim 256: 160 sub-head sequences
    (2, 200, 80, 2, 64, 32),    # headdim 32
]


@pytest.mark.parametrize("B,L,H,G,N,P", HANDOVER)
def test_ssd_bwd_handover_parity(B, L, H, G, N, P):
    x = _problem(B, L, H, G, N, seed=B + L + H + P, P=P)
    _, _, _, g = _gpu(_dev(x))
    if P > 64:
        _compare_wide(g, x, P)
    else:
        _compare(g, _oracle(x))


def test_ssd_bwd_handover_is_the_per_batch_result():
    """Two batch rows of 80 heads (160 sequences: ranges per SM, cut
    sequences) against each row alone (80 sequences: one CTA each, nothing
    cut): the per-sequence results -- dx, ddt_raw, dBm, dCm, dh0 -- are the
    same bit for bit (the handed-over state gradient is the same f32 values);
    the sums over the batch, dA_log, ddt_bias, dDp, agree to rounding."""
    x = _problem(2, 200, 80, 2, 64, seed=41)
    xd = _dev(x)
    _, _, _, g = _gpu(xd)
    parts = []
    for b in range(2):
        xb = {k: (v[b:b + 1].contiguous() if k in ("x", "dt_raw", "Bm", "Cm", "dy", "h0", "dh_last") else v)
              for k, v in xd.items()}
        _, _, _, gb = _gpu(xb)
        parts.append(gb)
        for k in ("dx", "ddt_raw", "dBm", "dCm", "dh0"):
            assert torch.equal(g[k][b:b + 1], gb[k]), (b, k)
    for k in ("dA_log", "ddt_bias", "dDp"):
        tot = np64(parts[0][k]) + np64(parts[1][k])
        assert np.allclose(np64(g[k]), tot, rtol=1e-5, atol=1e-6 * np.abs(tot).max()), k


def test_ssd_bwd_handover_dt_limit():
    """The limit on delta with sequences cut between CTAs."""
    x = _problem(2, 200, 80, 2, 64, seed=43)
    sp = torch.nn.functional.softplus(x["dt_raw"].double() + x["dt_bias"].double())
    lim = (float(np.float32(torch.quantile(sp.flatten()[::7].float(), 0.25))),
           float(np.float32(torch.quantile(sp.flatten()[::7].float(), 0.75))))
    _, _, _, g = _gpu(_dev(x), dt_limit=lim)
    _compare(g, _oracle(x, dt_limit=lim))


def test_ssd_bwd_handover_deterministic():
    xd = _dev(_problem(2, 300, 80, 2, 128, seed=13))
    _, _, cs, g0 = _gpu(xd)
    keep = {k: v.clone() for k, v in g0.items() if v is not None}
    for _ in range(4):
        g = s6.ssd_bwd(*[xd[k] for k in KEYS], cs, xd["dy"], xd["dh_last"])
        for k, v in keep.items():
            assert torch.equal(g[k], v), k


HEAD32 = [
    # B, L, H, G, N: headdim 32, run as 64 columns whose last 32 are zero
    (2, 200, 4, 2, 64),
    (1, 130, 3, 1, 128),
    (1, 1000, 8, 2, 128),   # few sequences: the forward cuts each in two
]


@pytest.mark.parametrize("B,L,H,G,N", HEAD32)
@pytest.mark.parametrize("variant", ["h0_dh", "plain"])
def test_ssd_bwd_head32(B, L, H, G, N, variant):
    full = variant == "h0_dh"
    x = _problem(B, L, H, G, N, seed=B + L + N + 32, h0=full, dh=full, P=32)
    y, h_last, cs, g = _gpu(_dev(x))
    assert cs.shape == (B, H, -(-L // 64), N, 32)
    ry, rh = oracle.ssd_fwd(*[x[k] for k in KEYS], x["h0"])
    assert rel_err(np64(y), ry) <= TOL["bf16"] and rel_err(np64(h_last), rh) <= TOL["bf16"]
    _compare(g, _oracle(x))


@pytest.mark.parametrize("B,L,H,G,N", [(2, 200, 4, 2, 64), (1, 1000, 8, 2, 128)])
def test_ssd_head32_is_head64_with_zero_columns(B, L, H, G, N):
    """Headdim 32 gives, bit for bit, what headdim 64 gives on the same problem
    with columns 32..63 of x, dy, h0 and dh_last set to zero: the same
    arithmetic on the same operands (the padding adds exact zeros), nothing
    written past column 32; and the padded run's own columns 32..63 of y,
    h_last, the saves, dx and dh0 are zero."""
    x32 = _problem(B, L, H, G, N, seed=77 + L, P=32)
    pad = lambda t: torch.nn.functional.pad(t, (0, 32))  # noqa: E731
    x64 = dict(x32, x=pad(x32["x"]), dy=pad(x32["dy"]), h0=pad(x32["h0"]), dh_last=pad(x32["dh_last"]))
    y32, hl32, cs32, g32 = _gpu(_dev(x32))
    y64, hl64, cs64, g64 = _gpu(_dev(x64))
    for a, b in ((y32, y64), (hl32, hl64), (cs32, cs64), (g32["dx"], g64["dx"]), (g32["dh0"], g64["dh0"])):
        assert torch.equal(a, b[..., :32].contiguous())
        assert not b[..., 32:].any()
    for k in ("ddt_raw", "ddt_bias", "dA_log", "dBm", "dCm", "dDp"):
        assert torch.equal(g32[k], g64[k]), k


WIDE = [
    # B, L, H, G, N, P: heads of 64 m columns run as m sub-heads
    (2, 200, 4, 2, 64, 128),
    (1, 130, 3, 1, 128, 192),
    (1, 300, 2, 1, 128, 256),
    (2, 64, 2, 2, 128, 128),    # exactly one chunk
]


@pytest.mark.parametrize("B,L,H,G,N,P", WIDE)
@pytest.mark.parametrize("variant", ["h0_dh", "plain"])
def test_ssd_bwd_wide_heads(B, L, H, G, N, P, variant):
    """Headdim 128..256: every gradient (ddt_raw, dA_log, ddt_bias, dDp summed
    over the head's sub-heads in a fixed order) against the oracle."""
    full = variant == "h0_dh"
    x = _problem(B, L, H, G, N, seed=B + L + P, h0=full, dh=full, P=P)
    _, _, cs, g = _gpu(_dev(x))
    assert cs.shape == (B, H, -(-L // 64), N, P)
    _compare_wide(g, x, P)


def test_ssd_bwd_wide_heads_deterministic():
    xd = _dev(_problem(2, 300, 4, 2, 128, seed=9, P=128))
    _, _, cs, g0 = _gpu(xd)
    keep = {k: v.clone() for k, v in g0.items() if v is not None}
    for _ in range(4):
        g = s6.ssd_bwd(*[xd[k] for k in KEYS], cs, xd["dy"], xd["dh_last"])
        for k, v in keep.items():
            assert torch.equal(g[k], v), k


def test_ssd_save_matches_plain_forward_and_the_oracle_states():
    """The saving forward gives the same y / h_last bit for bit as the plain
    one; chunk c of the saves is the state before step 64c (bf16)."""
    x = _problem(2, 200, 4, 2, 128, seed=3)
    xd = _dev(x)
    y0, h0 = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"])
    y1, h1, cs = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"], save=True)
    s6.check_device_status()
    assert torch.equal(y0, y1) and torch.equal(h0, h1)
    assert cs.shape == (2, 4, 4, 128, 64) and cs.dtype == torch.bfloat16
    assert torch.equal(cs[:, :, 0], xd["h0"].to(torch.bfloat16))
    for c in (1, 3):
        sub = {k: (v[:, : 64 * c].contiguous() if k in ("x", "dt_raw", "Bm", "Cm") else v) for k, v in x.items()}
        _, hc = oracle.ssd_fwd(*[sub[k] for k in KEYS], sub["h0"])
        assert rel_err(np64(cs[:, :, c]), hc) <= TOL["bf16"], c


def test_ssd_bwd_dt_limit():
    """A limit that clamps about half the steps: no gradient to dt_raw there."""
    x = _problem(2, 150, 4, 1, 128, seed=5)
    sp = torch.nn.functional.softplus(x["dt_raw"].double() + x["dt_bias"].double())
    lim = (float(np.float32(torch.quantile(sp.flatten()[::7].float(), 0.25))),
           float(np.float32(torch.quantile(sp.flatten()[::7].float(), 0.75))))
    _, _, _, g = _gpu(_dev(x), dt_limit=lim)
    ref = _oracle(x, dt_limit=lim)
    free = _oracle(x)
    assert rel_err(ref["ddt_raw"], free["ddt_raw"]) > 0.05  # the limit changes the answer
    _compare(g, ref)
    # clamped steps (softplus strictly outside the limit, away from the bounds) get exactly 0
    spn = sp.numpy()
    outside = (spn < lim[0] * 0.999) | (spn > lim[1] * 1.001)
    assert outside.any() and np.all(np64(g["ddt_raw"])[outside] == 0.0)


def test_ssd_bwd_steep_and_mixed_decays():
    x = _problem(2, 260, 6, 2, 128, seed=31)
    sp_inv = lambda v: float(np.log(np.expm1(v)))  # noqa: E731
    x["dt_bias"] = torch.tensor([sp_inv(3.0), sp_inv(1.0), sp_inv(0.05), sp_inv(6.0), sp_inv(0.9), sp_inv(0.01)],
                                dtype=torch.float32)
    x["A_log"] = torch.log(torch.tensor([16.0, 8.0, 4.0, 2.0, 9.0, 1.0], dtype=torch.float32))
    _, _, _, g = _gpu(_dev(x))
    ref = _oracle(x)
    _compare(g, ref)
    for h in range(6):
        assert rel_err(np64(g["dx"])[:, :, h], ref["dx"][:, :, h]) <= TOL["bf16"], h


def test_ssd_bwd_bitwise_deterministic_10_runs():
    xd = _dev(_problem(2, 500, 8, 2, 128, seed=7))
    _, _, cs, g0 = _gpu(xd)
    keep = {k: v.clone() for k, v in g0.items() if v is not None}
    for _ in range(9):
        g = s6.ssd_bwd(*[xd[k] for k in KEYS], cs, xd["dy"], xd["dh_last"])
        for k, v in keep.items():
            assert torch.equal(g[k], v), k


def test_ssd_bwd_empty_sequence():
    """No steps: the final-state gradient passes straight to dh0, the parameter
    gradients are zero."""
    xd = _dev(_problem(2, 0, 2, 1, 64, seed=1))
    _, _, cs = s6.ssd_fwd(*[xd[k] for k in KEYS], xd["h0"], save=True)
    g = s6.ssd_bwd(*[xd[k] for k in KEYS], cs, xd["dy"], xd["dh_last"])
    torch.cuda.synchronize()
    assert torch.equal(g["dh0"], xd["dh_last"])
    for k in ("ddt_bias", "dA_log", "dDp"):
        assert torch.count_nonzero(g[k]) == 0


def test_ssd_bwd_full_shape():
    """The Mamba-2-1.3B shape (B=4, L=4096, H=64, P=64, G=1, N=128): per-head
    gradients of sampled heads against the oracle run on those heads over
    every batch row; dBm and dCm (sums over all 64 heads) through
      sum dBm * Bm = sum_h (dx - D dy) . x   and   sum dCm * Cm = sum_h dy . (y - D x),
    which the chain rule gives at any size."""
    w = inputs.SSD_WORKLOADS["mamba2_1p3b"]
    x = _problem(w.batch, w.seqlen, w.nheads, w.ngroups, w.dstate, seed=0, h0=False, dh=False)
    xd = _dev(x)
    y, _, _, g = _gpu(xd)
    for h in (0, 37, 63):
        sub = {"x": x["x"][:, :, h:h + 1].contiguous(), "dt_raw": x["dt_raw"][:, :, h:h + 1].contiguous(),
               "dt_bias": x["dt_bias"][h:h + 1], "A_log": x["A_log"][h:h + 1], "Bm": x["Bm"], "Cm": x["Cm"],
               "Dp": x["Dp"][h:h + 1], "h0": None, "dy": x["dy"][:, :, h:h + 1].contiguous(), "dh_last": None}
        ref = _oracle(sub)
        assert rel_err(np64(g["dx"][:, :, h:h + 1]), ref["dx"]) <= TOL["bf16"], h
        assert rel_err(np64(g["ddt_raw"][:, :, h:h + 1]), ref["ddt_raw"]) <= TOL["bf16"], h
        assert rel_err(np64(g["dh0"][:, h:h + 1]), ref["dh0"]) <= TOL["bf16"], h
        for k in ("dA_log", "ddt_bias", "dDp"):
            assert rel_err(np64(g[k][h:h + 1]), ref[k]) <= TOL["bf16"], (h, k)
    D = xd["Dp"].double().view(1, 1, -1, 1)
    xs, dys, ys = xd["x"].double(), xd["dy"].double(), y.double()
    lhs_b = (g["dBm"].double() * xd["Bm"].double()).sum()
    rhs_b = ((g["dx"].double() - D * dys) * xs).sum()
    scale_b = (g["dBm"].double() * xd["Bm"].double()).abs().sum()
    assert abs(float(lhs_b - rhs_b)) <= 2e-2 * float(scale_b)
    lhs_c = (g["dCm"].double() * xd["Cm"].double()).sum()
    rhs_c = (dys * (ys - D * xs)).sum()
    scale_c = (g["dCm"].double() * xd["Cm"].double()).abs().sum()
    assert abs(float(lhs_c - rhs_c)) <= 2e-2 * float(scale_c)
    # bit-identical on repeat at full size
    g2 = s6.ssd_bwd(*[xd[k] for k in KEYS], s6.ssd_fwd(*[xd[k] for k in KEYS], None, save=True)[2], xd["dy"], None)
    for k in GRADS:
        assert torch.equal(g[k], g2[k]), k


def _sweep(n=8, seed=4321):
    r = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B = int(r.integers(1, 4))
        L = int(r.integers(1, 300))
        G = int(r.integers(1, 3))
        H = G * int(r.integers(1, 4))
        N = int(r.choice([64, 128]))
        out.append((B, L, H, G, N, bool(r.integers(0, 2)), bool(r.integers(0, 2))))
    return out


@pytest.mark.parametrize("B,L,H,G,N,with_state,limited", _sweep())
def test_ssd_bwd_random_shape_sweep(B, L, H, G, N, with_state, limited):
    x = _problem(B, L, H, G, N, seed=B * 11 + L, h0=with_state, dh=with_state)
    lim = (0.01, 0.05) if limited else None
    _, _, _, g = _gpu(_dev(x), dt_limit=lim)
    _compare(g, _oracle(x, dt_limit=lim))


def _handover_sweep(n=6, seed=2718):
    """Shapes with more (batch, sub-head) sequences than SMs (153..320): one
    range of chunks per SM, sequences cut and handed over (or, with one
    chunk each, never cut)."""
    r = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        B = int(r.integers(1, 4))
        G = int(r.integers(1, 3))
        P = int(r.choice([32, 64, 128]))
        m = max(1, P // 64)
        H = G * int(r.integers(1, 200))
        if not 152 < B * H * m <= 320:
            continue
        L = int(r.integers(1, 200))
        N = int(r.choice([64, 128]))
        out.append((B, L, H, G, N, P, bool(r.integers(0, 2)), bool(r.integers(0, 2))))
    return out


@pytest.mark.parametrize("B,L,H,G,N,P,with_state,limited", _handover_sweep())
def test_ssd_bwd_handover_random_sweep(B, L, H, G, N, P, with_state, limited):
    x = _problem(B, L, H, G, N, seed=B * 17 + L + H, h0=with_state, dh=with_state, P=P)
    lim = (0.01, 0.05) if limited else None
    _, _, _, g = _gpu(_dev(x), dt_limit=lim)
    if P > 64:
        _compare_wide(g, x, P, dt_limit=lim)
    else:
        _compare(g, _oracle(x, dt_limit=lim))


def _wide_sweep(n=6, seed=97):
    r = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B = int(r.integers(1, 3))
        L = int(r.integers(1, 260))
        G = int(r.integers(1, 3))
        H = G * int(r.integers(1, 3))
        N = int(r.choice([64, 128]))
        P = int(r.choice([128, 192, 256]))
        out.append((B, L, H, G, N, P, bool(r.integers(0, 2)), bool(r.integers(0, 2))))
    return out


@pytest.mark.parametrize("B,L,H,G,N,P,with_state,limited", _wide_sweep())
def test_ssd_bwd_wide_random_sweep(B, L, H, G, N, P, with_state, limited):
    x = _problem(B, L, H, G, N, seed=B * 13 + L + P, h0=with_state, dh=with_state, P=P)
    lim = (0.01, 0.05) if limited else None
    _, _, _, g = _gpu(_dev(x), dt_limit=lim)
    _compare_wide(g, x, P, dt_limit=lim)
