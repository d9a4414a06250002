"""ssm_scan_bwd_noalloc, checked against ssm_scan_bwd through the C ABI.

Some callers cannot allocate device memory: a host framework that owns the
device allocator and forbids raw cudaMalloc, a plugin interface that passes
only input and output pointers, a loop that must not allocate or synchronise.
ssm_scan_bwd_noalloc serves them by taking its scratch from a fixed array
inside the library instead of a caller buffer.  These tests call it twice in
a row (a larger problem, then a smaller one, so stale scratch from the first
call would show in the second) and require every gradient to equal the
regular entry point's bit for bit (both run the same kernels on the same
work plan, so any difference is a scratch error), and check that a shape
needing more scratch is refused.
"""
import ctypes

import pytest
import torch

from gpu_helpers import ARGS, np64, rel_err, to_dev
from selective_state_space_s6_gb300 import inputs, s6

pytestmark = pytest.mark.gpu

GRADS = ("du", "d_delta_raw", "dz", "dBm", "dCm", "dA_log", "dD", "d_delta_bias", "dh0")


def _lib():
    lib = s6.load_library()
    f = lib.ssm_scan_bwd_noalloc
    f.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int] + [ctypes.c_void_p] * 21 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    lib.ssm_noalloc_scratch_bytes.argtypes = []
    lib.ssm_noalloc_scratch_bytes.restype = ctypes.c_size_t
    return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, xd, cs, dh_last):
    B, L, D = xd["u"].shape
    N = xd["Bm"].shape[-1]
    act = s6.SSM_BF16 if xd["u"].dtype == torch.bfloat16 else s6.SSM_F32
    g = {
        "du": torch.empty_like(xd["u"]), "d_delta_raw": torch.empty_like(xd["u"]),
        "dz": torch.empty_like(xd["u"]), "dBm": torch.empty_like(xd["Bm"]),
        "dCm": torch.empty_like(xd["Cm"]), "dA_log": torch.empty_like(xd["A_log"]),
        "dD": torch.empty_like(xd["Dp"]), "d_delta_bias": torch.empty_like(xd["delta_bias"]),
        "dh0": torch.empty((B, D, N), dtype=torch.float32, device=xd["u"].device),
    }
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.ssm_scan_bwd_noalloc(
        B, L, D, N, act, *[_p(xd[k]) for k in ARGS], _p(xd["h0"]), _p(cs), _p(xd["dout"]),
        _p(dh_last), _p(g["du"]), _p(g["d_delta_raw"]), _p(g["dz"]), _p(g["dBm"]), _p(g["dCm"]),
        _p(g["dA_log"]), _p(g["dD"]), _p(g["d_delta_bias"]), _p(g["dh0"]), stream)
    assert rc == 0, (rc, lib.ssm_last_error().decode())
    return g


def test_noalloc_matches_regular_entry_point_on_two_calls_in_a_row():
    lib = _lib()
    cases = [(0, (2, 300, 130, 16, "bf16")), (1, (1, 97, 72, 16, "f32"))]
    for seed, shape in cases:
        x = inputs.make_inputs(*shape, seed=seed, h0_std=0.5, with_dh_last=True)
        xd = to_dev(x)
        _, _, cs = s6.ssm_scan_fwd(*[xd[k] for k in ARGS], xd["h0"])
        ref = s6.ssm_scan_bwd(*[xd[k] for k in ARGS], xd["h0"], cs, xd["dout"], xd["dh_last"])
        got = _noalloc(lib, xd, cs, xd["dh_last"])
        s6.check_device_status()
        for k in GRADS:
            assert torch.equal(got[k], ref[k]), (shape, k, rel_err(np64(got[k]), np64(ref[k])))


def test_noalloc_refuses_shapes_beyond_its_scratch():
    lib = _lib()
    limit = lib.ssm_noalloc_scratch_bytes()
    assert limit == 16 << 20
    B, L, D, N = 4, 4096, 4096, 16
    assert s6.bwd_workspace_bytes(B, L, D, N, s6.SSM_BF16) > limit
    fake = ctypes.c_void_p(0x10000)  # refused before any pointer is used
    rc = lib.ssm_scan_bwd_noalloc(B, L, D, N, s6.SSM_BF16, *([fake] * 21), None)
    assert rc == 2  # SSM_ERR_UNSUPPORTED
    assert b"scratch" in lib.ssm_last_error()
