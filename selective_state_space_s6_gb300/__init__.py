"""GB300-native S6 selective scan (Mamba) — forward, backward and decode step.

The compute path is the C-ABI library ``libssm_s6.so`` (hand-written CUDA for
sm_103a, declared in ``include/ssm_scan.h``); ``s6`` is its thin Python binding.
"""
from . import inputs  # noqa: F401  (seeded synthetic workloads; no CUDA needed)

__all__ = ["inputs"]
