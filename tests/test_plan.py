"""The persistent backward's work plan, checked on the host over many shapes
(no GPU): tests/plan_check.cu walks every CTA range item by item through the
plan helpers the kernels use and checks coverage, piece order, balance and the
aggregate pass's sub-pieces.  Also pins how short the split layout keeps the
aggregated tails on the Mamba-1.4B and Mamba-130m shapes."""
import os
import subprocess

import pytest

from selective_state_space_s6_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))

SHAPES = [
    # B, L, D, N
    (4, 4096, 4096, 16),    # Mamba-1.4B: 128 sequences on 152 CTAs (split layout)
    (8, 2048, 1536, 16),    # Mamba-130m (split layout)
    (4, 256, 5120, 16),     # hand-over shape (contiguous, two pieces)
    (2, 4096, 9728, 16),    # one sequence per CTA
    (16, 4096, 4096, 16),   # more sequences than CTAs (contiguous)
    (1, 65536, 2048, 16),   # a few very long sequences
    (1, 1100, 64, 16),      # one sequence over 35 CTAs
    (3, 5000, 200, 8),
    (1, 33, 128, 16),       # ragged: a head of one chunk
    (2, 4096, 4096, 16),
    (5, 100000, 256, 16),
    (7, 3000, 640, 4),
]


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    lib = build.build()
    exe = str(tmp_path_factory.mktemp("plan") / "plan_check")
    libdir = os.path.dirname(lib)
    cmd = [build.nvcc(), "-std=c++17", "-O1", f"-I{build.INCLUDE}", f"-I{build.CSRC}",
           os.path.join(HERE, "plan_check.cu"), "-o", exe, f"-L{libdir}", "-lssm_s6",
           "-Xlinker", f"-rpath={libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _run(exe, *shape, sms=152):
    r = subprocess.run([exe, *map(str, shape), str(sms)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr
    U, P, H, maxp, agg = map(int, r.stdout.split()[1:])
    return U, P, H, maxp, agg


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("sms", [152, 148, 7])
def test_plan_covers_and_balances(checker, shape, sms):
    _run(checker, *shape, sms=sms)


def test_split_layout_keeps_tails_short(checker):
    # Mamba-1.4B: 128 sequences of 128 chunks on 152 CTAs.  Heads of
    # ceil(16384 / 152) = 108 chunks; every tail of 20 chunks is aggregated,
    # 2560 chunks in all (the contiguous layout would aggregate 9120).
    assert _run(checker, 4, 4096, 4096, 16) == (16384, 152, 108, 3, 2560)
    # Mamba-130m: 96 sequences of 64 chunks; heads of 41, tails of 23
    U, P, H, maxp, agg = _run(checker, 8, 2048, 1536, 16)
    assert (U, P, H, agg) == (6144, 152, 41, 96 * 23)
    # as many sequences as CTAs: one sequence each, nothing aggregated
    assert _run(checker, 2, 4096, 9728, 16)[2:] == (0, 1, 0)
