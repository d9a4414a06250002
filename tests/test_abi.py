"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, and its host-only calls (status strings, sizes, argument
validation that fails before any launch) behave as documented."""
import ctypes
import os
import re

import pytest

from selective_state_space_s6_gb300 import build, s6

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm_scan.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return s6.load_library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for f in ("ssm_scan_fwd", "ssm_scan_fwd_nosave", "ssm_scan_bwd", "ssm_step"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(s6.library_path())
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, f"not exported: {missing}"


def test_status_strings_and_sizes(lib):
    assert lib.ssm_status_string(0) == b"SSM_OK"
    assert lib.ssm_status_string(3) == b"SSM_ERR_WORKSPACE"
    assert lib.ssm_status_string(99) == b"SSM_ERR_UNKNOWN"
    assert lib.ssm_version() >= 100
    c = s6.CHUNK_LEN
    assert [lib.ssm_num_chunks(x) for x in (0, 1, c, c + 1, 4096)] == [0, 1, 1, 2, 4096 // c]
    assert lib.ssm_fwd_workspace_bytes(1, 64, 16, 4, 0) == 0
    ws = lib.ssm_bwd_workspace_bytes(4, 4096, 4096, 16, 1)
    # per-64-channel-tile dBm/dCm partials plus per-batch parameter partials
    assert ws >= 64 * 4 * 4096 * 2 * 16 * 4 + 4 * 4096 * 18 * 4
    assert ws % 256 == 0
    assert lib.ssm_bwd_workspace_bytes(1, 8, 8, 0, 0) == -1
    assert lib.ssm_bwd_workspace_bytes(1, 8, 8, 4, 7) == -1


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails validation first


def _fwd(lib, B=1, L=8, D=8, N=4, act=0, **over):
    args = dict(u=FAKE, delta_raw=FAKE, z=None, Bm=FAKE, Cm=FAKE, A_log=FAKE, Dp=FAKE,
                delta_bias=FAKE, h0=None, out=FAKE, h_last=None, chunk_states=FAKE)
    args.update(over)
    return lib.ssm_scan_fwd(B, L, D, N, act, *args.values(), None, 0, None)


def test_fwd_argument_validation(lib):
    assert _fwd(lib, N=0) == 1
    assert _fwd(lib, N=17) == 2
    assert _fwd(lib, B=-1) == 1
    assert _fwd(lib, act=5) == 1
    assert _fwd(lib, u=None) == 1
    assert b"u must not be NULL" in lib.ssm_last_error()
    assert _fwd(lib, chunk_states=None) == 1
    assert _fwd(lib, Bm=ctypes.c_void_p(0x10002)) == 1  # f32 needs 4-byte alignment
    assert b"aligned" in lib.ssm_last_error()


def test_bwd_workspace_and_gradient_checks(lib):
    B, L, D, N = 2, 16, 8, 4
    need = lib.ssm_bwd_workspace_bytes(B, L, D, N, 0)
    ptrs = [FAKE] * 21
    # z given (index 2) but dz (index 14) missing -> invalid argument
    p = list(ptrs)
    p[14] = None
    assert lib.ssm_scan_bwd(B, L, D, N, 0, *p, FAKE, need, None) == 1
    assert b"dz" in lib.ssm_last_error()
    # workspace too small
    assert lib.ssm_scan_bwd(B, L, D, N, 0, *ptrs, FAKE, need - 4, None) == 3
    assert lib.ssm_scan_bwd(B, L, D, N, 0, *ptrs, None, need, None) == 3


def test_step_validation(lib):
    args = [FAKE] * 10
    args[8] = None  # h
    assert lib.ssm_step(2, 8, 4, 0, *args, None) == 1
    assert b"h must not be NULL" in lib.ssm_last_error()


def test_dt_limit_validation(lib):
    """The _ex entry points check the limit first: 0 <= dt_min <= dt_max."""
    def opts(lo, hi):
        return ctypes.byref(s6.ScanOptions(lo, hi))

    fwd12 = [FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE]
    for lo, hi in ((0.5, 0.1), (-0.1, 1.0), (float("nan"), 1.0), (0.0, float("nan"))):
        assert lib.ssm_scan_fwd_ex(1, 8, 8, 4, 0, *fwd12, None, 0, None, opts(lo, hi)) == 1
        assert b"dt limit" in lib.ssm_last_error()
        assert lib.ssm_scan_bwd_ex(2, 16, 8, 4, 0, *([FAKE] * 21), FAKE, 1 << 20, None, opts(lo, hi)) == 1
        assert lib.ssm_scan_bwd_partials_ex(2, 16, 8, 4, 0, *([FAKE] * 15), FAKE, 1 << 20, None,
                                            opts(lo, hi)) == 1
        assert lib.ssm_step_ex(2, 8, 4, 0, *([FAKE] * 10), None, opts(lo, hi)) == 1
        assert b"dt limit" in lib.ssm_last_error()
    # accepted limits (equal ends, an infinite top, none at all) reach the next check
    for o in (opts(0.25, 0.25), opts(0.0, float("inf")), None):
        bad = list(fwd12)
        bad[0] = None
        assert lib.ssm_scan_fwd_ex(1, 8, 8, 4, 0, *bad, None, 0, None, o) == 1
        assert b"u must not be NULL" in lib.ssm_last_error()


def test_ssd_validation(lib):
    """Host-side checks of ssm_ssd_fwd: unsupported shapes and dtypes, groups
    that do not divide the heads, misaligned tensors -- all before any launch."""
    args = [FAKE] * 10
    def call(B=1, L=8, H=2, P=64, G=1, N=64, act=1, a=None):
        return lib.ssm_ssd_fwd(B, L, H, P, G, N, act, *(a or args), None, None)
    assert call(P=16) == 2 and b"headdim 32 or a multiple of 64" in lib.ssm_last_error()
    assert call(P=48) == 2                       # neither 32 nor 64 m columns
    assert call(P=96) == 2 and call(P=320) == 2  # 64 m columns, m <= 4
    assert call(N=16) == 2
    assert call(act=0) == 2                      # f32 activations: not built
    assert call(H=3, G=2) == 1 and b"multiple of ngroups" in lib.ssm_last_error()
    bad = list(args)
    bad[0] = ctypes.c_void_p(0x10008)            # x only 8-byte aligned
    assert call(a=bad) == 1 and b"x is not 16-byte aligned" in lib.ssm_last_error()


def test_segment_plan(lib):
    """The plans are functions of the shape.  Forward: one pass where the grid
    fills the GPU, time segments of at least 512 steps for long sequences over
    few channels.  Backward: the (batch x 128-channel tile) sequences are cut
    into 152 equal ranges of 32-step chunks; it reports 1 when no aggregate
    pass is needed (no cut, or cut sequences hand their carry over), else the
    most pieces any sequence has."""
    bf16, f32 = s6.SSM_BF16, s6.SSM_F32
    # 4 x 32 sequences of 128 chunks over 152 ranges of ~108 chunks: ranges
    # shorter than a sequence, some sequences cut twice: aggregate pass
    assert s6.plan_segments(4, 4096, 4096, 16, bf16) == (1, 3)
    # 4 x 40 sequences of 8 chunks over 152 ranges of ~8.4 chunks: at most one
    # cut each, ranges longer than a sequence: carries handed over
    assert s6.plan_segments(4, 256, 5120, 16, bf16)[1] == 1
    # 152 sequences: one range each, no cut
    assert s6.plan_segments(2, 4096, 76 * 128, 16, bf16)[1] == 1
    # one sequence of 35 chunks: 35 ranges of one chunk
    assert s6.plan_segments(1, 1100, 64, 16, f32)[1] == -(-1100 // s6.CHUNK_LEN)
    f, b = s6.plan_segments(1, 65536, 2048, 16, f32)
    assert f > 1 and b > 1
    for shape in [(1, 64, 16, 4), (2, 1023, 64, 16), (3, 5000, 200, 8), (1, 4096, 32, 16)]:
        f, b = s6.plan_segments(*shape, f32)
        assert f >= 1 and b >= 1
        if f > 1:
            assert -(-shape[1] // f) >= 512
        assert s6.plan_segments(*shape, f32) == (f, b)
    # dstate outside {4, 8, 16} never cuts sequences (generic kernels)
    assert s6.plan_segments(3, 5000, 200, 5, f32)[1] == 1
    # short sequences are never split in time by the forward
    assert s6.plan_segments(1, 1000, 64, 16, f32)[0] == 1
    with pytest.raises(s6.SSMError):
        s6.plan_segments(1, 10, 16, 32, f32)  # dstate above 16


def test_ssd_bwd_validation(lib):
    """Host-side checks of ssm_ssd_bwd and its workspace query: unsupported
    shapes, misaligned tensors, a missing or short workspace -- before any
    launch."""
    assert lib.ssm_ssd_bwd_workspace_bytes(1, 8, 2, 64, 1, 16, 1) == -1   # dstate 16: not supported
    assert lib.ssm_ssd_bwd_workspace_bytes(1, 8, 3, 64, 2, 64, 1) == -1   # heads not a multiple of groups
    need = lib.ssm_ssd_bwd_workspace_bytes(2, 100, 4, 64, 2, 128, 1)
    assert need >= 2 * 2 * 100 * 4 * 128 * 4 and need % 256 == 0
    # headdim 128: two sub-heads per head -- twice the per-sub-head terms,
    # plus their ddt_raw terms
    need2 = lib.ssm_ssd_bwd_workspace_bytes(2, 100, 4, 128, 2, 128, 1)
    assert need2 >= 2 * 2 * 100 * 8 * 128 * 4 + 2 * 100 * 8 * 4 and need2 % 256 == 0
    assert lib.ssm_ssd_bwd_workspace_bytes(2, 100, 4, 96, 2, 128, 1) == -1
    # headdim 32: one sub-head per head (64 columns, the last 32 zero), the
    # workspace of headdim 64
    assert lib.ssm_ssd_bwd_workspace_bytes(2, 100, 4, 32, 2, 128, 1) == need
    assert lib.ssm_ssd_bwd_workspace_bytes(2, 100, 4, 16, 2, 128, 1) == -1
    args = [FAKE] * 19  # x .. dh0, ws

    def call(B=2, L=100, H=4, P=64, G=2, N=128, act=1, a=None, ws_bytes=None):
        return lib.ssm_ssd_bwd(B, L, H, P, G, N, act, *(a or args), need if ws_bytes is None else ws_bytes, None, None)
    assert call(N=32) == 2 and b"dstate 64 or 128" in lib.ssm_last_error()
    assert call(act=0) == 2
    bad = list(args)
    bad[8] = ctypes.c_void_p(0x10008)            # dy only 8-byte aligned
    assert call(a=bad) == 1 and b"dy is not 16-byte aligned" in lib.ssm_last_error()
    bad = list(args)
    bad[7] = None                                # chunk_states missing
    assert call(a=bad) == 1 and b"chunk_states must not be NULL" in lib.ssm_last_error()
    assert call(ws_bytes=need - 256) == 3        # SSM_ERR_WORKSPACE
