"""Seeded synthetic inputs for the S6 selective scan.

This module only draws random numbers in a fixed, documented order; it holds
none of the scan's arithmetic.  It is the one module that both the CUDA path's
tests/benchmark and the oracle's checks take their inputs from.

Recipe (every workload):
  * one ``torch.Generator`` on the CPU, ``manual_seed(seed)`` (seed 0 by default);
  * draw order: u, z, delta_raw, U (for delta_bias), Bm, Cm, dout, h0, dh_last;
  * u, z, delta_raw, Bm, Cm, dout ~ N(0, 1) in float32;
  * delta_bias[d] = log(expm1(U[d])), U ~ Uniform[lo, hi], so that
    softplus(delta_bias) = U (the usual Mamba dt initialisation);
  * A_log[d, n] = log(n + 1) (S4D-real initialisation, A = -(n+1));
  * Dp[d] = 1;
  * h0 ~ N(0, h0_std^2) when requested (the decode workload uses std 0.5);
  * dh_last ~ N(0, 1) when requested (gradient arriving at the final state);
  * activations (u, delta_raw, z, Bm, Cm, dout) are rounded once to bf16
    (round-to-nearest-even) when the workload is bf16; parameters and state
    stay float32.  Both sides then see exactly the same values.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes (B, L, D, N), activation dtype, Δ-bias range."""
    name: str
    batch: int
    seqlen: int
    dim: int
    dstate: int
    act: str  # "f32" or "bf16"
    delta_lo: float = 1e-3
    delta_hi: float = 0.1
    h0_std: Optional[float] = None
    description: str = ""

    @property
    def cells(self) -> int:
        return self.batch * self.seqlen * self.dim * self.dstate


WORKLOADS = {
    "tiny": Workload("tiny", 1, 64, 16, 4, "f32",
                     description="tiny S6 scan fwd+bwd, fp32: B=1 L=64 D=16 N=4"),
    "decode": Workload("decode", 256, 1000, 1536, 16, "f32", h0_std=0.5,
                       description="ssm_step decode, fp32: batch 256, d_inner 1536, N=16, "
                                   "1000 chained steps from h_prev ~ N(0, 0.5^2)"),
    "mamba130m": Workload("mamba130m", 8, 2048, 1536, 16, "bf16",
                          description="Mamba-130M-shaped scan fwd+bwd: B=8 L=2048 "
                                      "d_inner=1536 N=16, bf16 activations"),
    "mamba1p4b": Workload("mamba1p4b", 4, 4096, 4096, 16, "bf16",
                          description="Mamba-1.4B-shaped scan fwd+bwd: B=4 L=4096 "
                                      "d_inner=4096 N=16, bf16 activations"),
    "long": Workload("long", 1, 65536, 2048, 16, "f32", delta_lo=1e-4, delta_hi=1e-2,
                     description="long-sequence scan fwd+bwd, fp32: B=1 L=65536 "
                                 "d_inner=2048 N=16, softplus(delta_bias) in [1e-4, 1e-2]"),
}


def act_dtype(act: str) -> torch.dtype:
    if act == "f32":
        return torch.float32
    if act == "bf16":
        return torch.bfloat16
    raise ValueError(f"unknown activation dtype {act!r}")


def make_inputs(batch: int, seqlen: int, dim: int, dstate: int, act: str = "f32", *,
                seed: int = 0, delta_lo: float = 1e-3, delta_hi: float = 0.1,
                h0_std: Optional[float] = None, with_z: bool = True,
                with_dout: bool = True, with_dh_last: bool = False) -> dict:
    """Draw one problem on the CPU.  Returns a dict of tensors:

    u, delta_raw, z, dout : [B, L, D] (act dtype);  Bm, Cm : [B, L, N] (act dtype)
    A_log : [D, N], Dp : [D], delta_bias : [D] (float32);  h0, dh_last : [B, D, N] float32 or None
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    dt = act_dtype(act)
    bld = (batch, seqlen, dim)
    bln = (batch, seqlen, dstate)

    def normal(shape):
        return torch.randn(shape, generator=g, dtype=torch.float32)

    u = normal(bld)
    z = normal(bld)
    delta_raw = normal(bld)
    U = torch.rand((dim,), generator=g, dtype=torch.float64) * (delta_hi - delta_lo) + delta_lo
    Bm = normal(bln)
    Cm = normal(bln)
    dout = normal(bld)  # always drawn, so h0 comes from the same stream position
    if not with_dout:
        dout = None
    h0 = normal((batch, dim, dstate)) * h0_std if h0_std is not None else None
    dh_last = normal((batch, dim, dstate)) if with_dh_last else None

    delta_bias = torch.log(torch.expm1(U)).to(torch.float32)
    A_log = torch.log(torch.arange(1, dstate + 1, dtype=torch.float64)).to(torch.float32)
    A_log = A_log.unsqueeze(0).expand(dim, dstate).contiguous()
    Dp = torch.ones((dim,), dtype=torch.float32)

    cast = (lambda x: x.to(dt).contiguous()) if dt != torch.float32 else (lambda x: x.contiguous())
    return {
        "u": cast(u), "delta_raw": cast(delta_raw), "z": cast(z) if with_z else None,
        "Bm": cast(Bm), "Cm": cast(Cm), "A_log": A_log, "Dp": Dp, "delta_bias": delta_bias,
        "dout": cast(dout) if dout is not None else None, "h0": h0, "dh_last": dh_last,
    }


def make_workload(name: str, *, seed: int = 0, batch: Optional[int] = None,
                  seqlen: Optional[int] = None, with_dout: bool = True) -> dict:
    """Inputs for a named workload (optionally with fewer batches or steps)."""
    w = WORKLOADS[name]
    return make_inputs(batch or w.batch, seqlen or w.seqlen, w.dim, w.dstate, w.act, seed=seed,
                       delta_lo=w.delta_lo, delta_hi=w.delta_hi, h0_std=w.h0_std,
                       with_dout=with_dout)


# ------------------------------------------------------------------ Mamba-2 SSD

@dataclasses.dataclass(frozen=True)
class SsdWorkload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    ngroups: int
    dstate: int
    act: str
    description: str = ""

    @property
    def cells(self) -> int:
        return self.batch * self.seqlen * self.nheads * self.headdim * self.dstate


SSD_WORKLOADS = {
    "mamba2_1p3b": SsdWorkload("mamba2_1p3b", 4, 4096, 64, 64, 1, 128, "bf16",
                               description="Mamba-2-1.3B-shaped SSD forward: B=4 L=4096 heads=64 "
                                           "headdim=64 groups=1 N=128, bf16 activations"),
    # the same block width in heads of 128 columns (two sub-heads per head)
    "mamba2_1p3b_p128": SsdWorkload("mamba2_1p3b_p128", 4, 4096, 32, 128, 1, 128, "bf16",
                                    description="Mamba-2-1.3B width, headdim 128: B=4 L=4096 heads=32 "
                                                "headdim=128 groups=1 N=128, bf16 activations"),
}


def make_ssd_inputs(batch: int, seqlen: int, nheads: int, headdim: int, ngroups: int, dstate: int,
                    act: str = "bf16", *, seed: int = 0, h0_std: Optional[float] = None) -> dict:
    """Draw one SSD problem on the CPU (Mamba-2 initialisation: softplus(dt_bias)
    ~ U[1e-3, 0.1] and A = exp(A_log) ~ U[1, 16] per head, Dp = 1).  Returns
    x [B,L,H,P], dt_raw [B,L,H], Bm / Cm [B,L,G,N] (act dtype); dt_bias, A_log,
    Dp [H] and h0 [B,H,N,P] (or None) float32."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    dt = act_dtype(act)

    def normal(shape):
        return torch.randn(shape, generator=g, dtype=torch.float32)

    x = normal((batch, seqlen, nheads, headdim))
    dt_raw = normal((batch, seqlen, nheads))
    Bm = normal((batch, seqlen, ngroups, dstate))
    Cm = normal((batch, seqlen, ngroups, dstate))
    U = torch.rand((nheads,), generator=g, dtype=torch.float64) * (0.1 - 1e-3) + 1e-3
    Aval = torch.rand((nheads,), generator=g, dtype=torch.float64) * 15.0 + 1.0
    h0 = normal((batch, nheads, dstate, headdim)) * h0_std if h0_std is not None else None
    cast = (lambda v: v.to(dt).contiguous()) if dt != torch.float32 else (lambda v: v.contiguous())
    return {"x": cast(x), "dt_raw": cast(dt_raw), "Bm": cast(Bm), "Cm": cast(Cm),
            "dt_bias": torch.log(torch.expm1(U)).to(torch.float32), "A_log": torch.log(Aval).to(torch.float32),
            "Dp": torch.ones((nheads,), dtype=torch.float32), "h0": h0}
