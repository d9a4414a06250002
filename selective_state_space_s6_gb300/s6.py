"""Thin Python binding of the C-ABI library ``libssm_s6.so`` (include/ssm_scan.h).

Argument marshalling only: every step of the scan runs in the library's CUDA
kernels.  PyTorch supplies the device memory (output tensors are allocated
with ``torch.empty`` when not passed in) and the stream (the current torch
stream unless one is given).  There is no CPU fallback: if the library is
missing or a call fails, these functions raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libssm_s6.so")
_lock = threading.Lock()
_lib = None

SSM_F32, SSM_BF16 = 0, 1
CONV_PATHS = {0: "scalar", 1: "vector", 2: "tile"}
CHUNK_LEN = 32
MAX_DSTATE = 16


class ScanOptions(ctypes.Structure):
    """``ssm_scan_options``: the limit [dt_min, dt_max] on delta."""
    _fields_ = [("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float)]


def _opts(dt_limit):
    """ctypes pointer to the options for ``dt_limit = (dt_min, dt_max)``."""
    return ctypes.byref(ScanOptions(float(dt_limit[0]), float(dt_limit[1])))


class SSMError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed: {code} ({msg})")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load ``libssm_s6.so`` (building it first if it is absent and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            from . import build as _build
            _build.build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, vp, ci, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.ssm_status_string.argtypes = [ci]
        lib.ssm_status_string.restype = ctypes.c_char_p
        lib.ssm_last_error.argtypes = []
        lib.ssm_last_error.restype = ctypes.c_char_p
        lib.ssm_version.argtypes = []
        lib.ssm_version.restype = ci
        lib.ssm_check_device_status.argtypes = [vp]
        lib.ssm_check_device_status.restype = ci
        lib.ssm_num_chunks.argtypes = [i64]
        lib.ssm_num_chunks.restype = i64
        for f in (lib.ssm_fwd_workspace_bytes, lib.ssm_bwd_workspace_bytes):
            f.argtypes = [i64, i64, i64, i64, ci]
            f.restype = i64
        lib.ssm_scan_fwd.argtypes = [i64] * 4 + [ci] + [vp] * 12 + [vp, sz, vp]
        lib.ssm_scan_fwd.restype = ci
        lib.ssm_scan_fwd_nosave.argtypes = [i64] * 4 + [ci] + [vp] * 11 + [vp, sz, vp]
        lib.ssm_scan_fwd_nosave.restype = ci
        lib.ssm_scan_bwd.argtypes = [i64] * 4 + [ci] + [vp] * 21 + [vp, sz, vp]
        lib.ssm_scan_bwd.restype = ci
        lib.ssm_scan_bwd_partials.argtypes = [i64] * 4 + [ci] + [vp] * 15 + [vp, sz, vp]
        lib.ssm_scan_bwd_partials.restype = ci
        lib.ssm_scan_bwd_finalize.argtypes = [i64] * 4 + [ci] + [vp] * 5 + [vp, sz, vp]
        lib.ssm_scan_bwd_finalize.restype = ci
        lib.ssm_step.argtypes = [i64] * 3 + [ci] + [vp] * 10 + [vp]
        lib.ssm_step.restype = ci
        op = ctypes.POINTER(ScanOptions)
        lib.ssm_scan_fwd_ex.argtypes = [i64] * 4 + [ci] + [vp] * 12 + [vp, sz, vp, op]
        lib.ssm_scan_fwd_ex.restype = ci
        lib.ssm_scan_bwd_ex.argtypes = [i64] * 4 + [ci] + [vp] * 21 + [vp, sz, vp, op]
        lib.ssm_scan_bwd_ex.restype = ci
        lib.ssm_scan_bwd_partials_ex.argtypes = [i64] * 4 + [ci] + [vp] * 15 + [vp, sz, vp, op]
        lib.ssm_scan_bwd_partials_ex.restype = ci
        lib.ssm_step_ex.argtypes = [i64] * 3 + [ci] + [vp] * 10 + [vp, op]
        lib.ssm_step_ex.restype = ci
        lib.ssm_ssd_fwd.argtypes = [i64] * 6 + [ci] + [vp] * 10 + [op, vp]
        lib.ssm_ssd_fwd.restype = ci
        lib.ssm_ssd_fwd_save.argtypes = [i64] * 6 + [ci] + [vp] * 11 + [op, vp]
        lib.ssm_ssd_fwd_save.restype = ci
        lib.ssm_ssd_bwd_workspace_bytes.argtypes = [i64] * 6 + [ci]
        lib.ssm_ssd_bwd_workspace_bytes.restype = i64
        lib.ssm_ssd_bwd.argtypes = [i64] * 6 + [ci] + [vp] * 19 + [sz, op, vp]
        lib.ssm_ssd_bwd.restype = ci
        lib.ssm_conv1d_fwd.argtypes = [i64] * 4 + [ci] + [vp] * 6 + [vp]
        lib.ssm_conv1d_fwd.restype = ci
        lib.ssm_conv1d_bwd_workspace_bytes.argtypes = [i64] * 4 + [ci]
        lib.ssm_conv1d_bwd_workspace_bytes.restype = i64
        lib.ssm_conv1d_bwd.argtypes = [i64] * 4 + [ci] + [vp] * 9 + [vp, sz, vp]
        lib.ssm_conv1d_bwd.restype = ci
        lib.ssm_conv1d_step.argtypes = [i64] * 3 + [ci] + [vp] * 5 + [vp]
        lib.ssm_conv1d_step.restype = ci
        lib.ssm_conv1d_path.argtypes = [i64] * 4 + [ci] + [vp] * 3
        lib.ssm_conv1d_path.restype = ci
        lib.ssm_selftest_wait_timeout.argtypes = [vp]
        lib.ssm_selftest_wait_timeout.restype = ci
        lib.ssm_plan_segments.argtypes = [i64] * 4 + [ci, ctypes.POINTER(ci), ctypes.POINTER(ci)]
        lib.ssm_plan_segments.restype = ci
        lib.ssm_plan_fallbacks.argtypes = []
        lib.ssm_plan_fallbacks.restype = i64
        _lib = lib
        return lib


def _check(fn, rc):
    if rc != 0:
        lib = load_library()
        raise SSMError(fn, lib.ssm_status_string(rc).decode(), lib.ssm_last_error().decode())


def _act(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSM_F32
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    raise TypeError(f"activation dtype must be float32 or bfloat16, got {t.dtype}")


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def num_chunks(seqlen: int) -> int:
    return int(load_library().ssm_num_chunks(seqlen))


def fwd_workspace_bytes(batch, seqlen, dim, dstate, act) -> int:
    return int(load_library().ssm_fwd_workspace_bytes(batch, seqlen, dim, dstate, act))


def bwd_workspace_bytes(batch, seqlen, dim, dstate, act) -> int:
    return int(load_library().ssm_bwd_workspace_bytes(batch, seqlen, dim, dstate, act))


def plan_segments(batch, seqlen, dim, dstate, act):
    """(forward, backward) time-segment counts of the chunked parallel scan for this shape."""
    f, b = ctypes.c_int(0), ctypes.c_int(0)
    _check("ssm_plan_segments", load_library().ssm_plan_segments(batch, seqlen, dim, dstate, act,
                                                                  ctypes.byref(f), ctypes.byref(b)))
    return f.value, b.value


def plan_fallbacks():
    """Calls so far whose cooperative plan mode (forward stream mode, backward
    hand-over mode) did not fit on the GPU and ran non-cooperatively instead."""
    return int(load_library().ssm_plan_fallbacks())


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor]):
    if nbytes <= 0:
        return ws, 0
    if ws is None:
        ws = torch.empty((nbytes + 256,), dtype=torch.uint8, device=device)
    # the library wants 256-byte alignment; torch's caching allocator gives 512
    if ws.numel() < nbytes or ws.data_ptr() % 256:
        raise ValueError("workspace too small or misaligned")
    return ws, ws.numel()


def ssm_scan_fwd(u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h0=None, *, out=None,
                 h_last=None, chunk_states=None, save=True, want_h_last=True, ws=None,
                 stream=None, dt_limit=None):
    """Forward scan.  Returns ``(out, h_last, chunk_states)`` (chunk_states None when
    ``save=False``).  Shapes as in include/ssm_scan.h.  ``dt_limit = (dt_min,
    dt_max)`` clamps delta (the ``_ex`` entry point)."""
    B, L, D = u.shape
    N = Bm.shape[-1]
    act = _act(u)
    dev = u.device
    if out is None:
        out = torch.empty_like(u)
    if h_last is None and want_h_last:
        h_last = torch.empty((B, D, N), dtype=torch.float32, device=dev)
    lib = load_library()
    ws, ws_bytes = _workspace(fwd_workspace_bytes(B, L, D, N, act), dev, ws)
    if save and chunk_states is None:
        chunk_states = torch.empty((B, num_chunks(L), D, N), dtype=torch.float32, device=dev)
    if dt_limit is not None:
        cs = chunk_states if save else None
        rc = lib.ssm_scan_fwd_ex(B, L, D, N, act, _p(u), _p(delta_raw), _p(z), _p(Bm), _p(Cm),
                                 _p(A_log), _p(Dp), _p(delta_bias), _p(h0), _p(out), _p(h_last),
                                 _p(cs), _p(ws), ws_bytes, _stream(stream), _opts(dt_limit))
        _check("ssm_scan_fwd_ex", rc)
        return out, h_last, cs
    if save:
        rc = lib.ssm_scan_fwd(B, L, D, N, act, _p(u), _p(delta_raw), _p(z), _p(Bm), _p(Cm),
                              _p(A_log), _p(Dp), _p(delta_bias), _p(h0), _p(out), _p(h_last),
                              _p(chunk_states), _p(ws), ws_bytes, _stream(stream))
        _check("ssm_scan_fwd", rc)
        return out, h_last, chunk_states
    rc = lib.ssm_scan_fwd_nosave(B, L, D, N, act, _p(u), _p(delta_raw), _p(z), _p(Bm), _p(Cm),
                                 _p(A_log), _p(Dp), _p(delta_bias), _p(h0), _p(out),
                                 _p(h_last), _p(ws), ws_bytes, _stream(stream))
    _check("ssm_scan_fwd_nosave", rc)
    return out, h_last, None


def ssm_scan_fwd_nosave(u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h0=None, **kw):
    out, h_last, _ = ssm_scan_fwd(u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h0,
                                  save=False, **kw)
    return out, h_last


def ssm_scan_bwd(u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h0, chunk_states, dout,
                 dh_last=None, *, grads=None, want_dh0=True, ws=None, stream=None, split=False,
                 dt_limit=None):
    """Backward.  Returns a dict with du, d_delta_raw, dz (None without z), dBm, dCm,
    dA_log, dD, d_delta_bias, dh0 (None unless ``want_dh0``).  Pass ``grads`` (a dict
    of preallocated tensors with those keys) to write into existing buffers."""
    B, L, D = u.shape
    N = Bm.shape[-1]
    act = _act(u)
    dev = u.device
    g = dict(grads) if grads else {}
    g.setdefault("du", torch.empty_like(u))
    g.setdefault("d_delta_raw", torch.empty_like(u))
    g.setdefault("dz", torch.empty_like(u) if z is not None else None)
    g.setdefault("dBm", torch.empty_like(Bm))
    g.setdefault("dCm", torch.empty_like(Cm))
    g.setdefault("dA_log", torch.empty_like(A_log))
    g.setdefault("dD", torch.empty_like(Dp))
    g.setdefault("d_delta_bias", torch.empty_like(delta_bias))
    g.setdefault("dh0", torch.empty((B, D, N), dtype=torch.float32, device=dev) if want_dh0 else None)
    lib = load_library()
    ws, ws_bytes = _workspace(bwd_workspace_bytes(B, L, D, N, act), dev, ws)
    if split:
        bwd_partials(u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, chunk_states, dout, dh_last,
                     g, ws, stream, dt_limit=dt_limit)
        bwd_finalize(B, L, D, N, act, g, ws, stream)
        return g
    if dt_limit is not None:
        rc = lib.ssm_scan_bwd_ex(B, L, D, N, act, _p(u), _p(delta_raw), _p(z), _p(Bm), _p(Cm),
                                 _p(A_log), _p(Dp), _p(delta_bias), _p(h0), _p(chunk_states),
                                 _p(dout), _p(dh_last), _p(g["du"]), _p(g["d_delta_raw"]),
                                 _p(g["dz"]), _p(g["dBm"]), _p(g["dCm"]), _p(g["dA_log"]),
                                 _p(g["dD"]), _p(g["d_delta_bias"]), _p(g["dh0"]), _p(ws), ws_bytes,
                                 _stream(stream), _opts(dt_limit))
        _check("ssm_scan_bwd_ex", rc)
        return g
    rc = lib.ssm_scan_bwd(B, L, D, N, act, _p(u), _p(delta_raw), _p(z), _p(Bm), _p(Cm),
                          _p(A_log), _p(Dp), _p(delta_bias), _p(h0), _p(chunk_states),
                          _p(dout), _p(dh_last), _p(g["du"]), _p(g["d_delta_raw"]),
                          _p(g["dz"]), _p(g["dBm"]), _p(g["dCm"]), _p(g["dA_log"]),
                          _p(g["dD"]), _p(g["d_delta_bias"]), _p(g["dh0"]), _p(ws), ws_bytes,
                          _stream(stream))
    _check("ssm_scan_bwd", rc)
    return g


def bwd_partials(u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, chunk_states, dout, dh_last,
                 g, ws, stream=None, dt_limit=None):
    """First half of the backward (the scan); ``g`` holds preallocated outputs."""
    B, L, D = u.shape
    N = Bm.shape[-1]
    args = (B, L, D, N, _act(u), _p(u), _p(delta_raw), _p(z), _p(Bm), _p(Cm), _p(A_log), _p(Dp),
            _p(delta_bias), _p(chunk_states), _p(dout), _p(dh_last), _p(g["du"]),
            _p(g["d_delta_raw"]), _p(g["dz"]), _p(g.get("dh0")), _p(ws),
            0 if ws is None else ws.numel(), _stream(stream))
    if dt_limit is not None:
        _check("ssm_scan_bwd_partials_ex", load_library().ssm_scan_bwd_partials_ex(*args, _opts(dt_limit)))
        return
    rc = load_library().ssm_scan_bwd_partials(*args)
    _check("ssm_scan_bwd_partials", rc)


def bwd_finalize(B, L, D, N, act, g, ws, stream=None):
    """Second half of the backward: fixed-order sums of the partials left in ``ws``."""
    rc = load_library().ssm_scan_bwd_finalize(
        B, L, D, N, act, _p(g["dBm"]), _p(g["dCm"]), _p(g["dA_log"]), _p(g["dD"]),
        _p(g["d_delta_bias"]), _p(ws), 0 if ws is None else ws.numel(), _stream(stream))
    _check("ssm_scan_bwd_finalize", rc)


def ssm_step(u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h, *, out=None, stream=None,
             dt_limit=None):
    """One decode step; ``h`` [B,D,N] f32 is updated in place.  Returns ``out`` [B,D]."""
    B, D = u.shape
    N = Bm.shape[-1]
    act = _act(u)
    if out is None:
        out = torch.empty_like(u)
    args = (B, D, N, act, _p(u), _p(delta_raw), _p(z), _p(Bm), _p(Cm), _p(A_log), _p(Dp),
            _p(delta_bias), _p(h), _p(out), _stream(stream))
    if dt_limit is not None:
        _check("ssm_step_ex", load_library().ssm_step_ex(*args, _opts(dt_limit)))
        return out
    rc = load_library().ssm_step(*args)
    _check("ssm_step", rc)
    return out


def selftest_wait_timeout(stream=None):
    """Enqueue the library's give-up self-test (a bounded wait that runs out
    after ~2 s); the next check_device_status() raises with SSM_ERR_TIMEOUT."""
    _check("ssm_selftest_wait_timeout", load_library().ssm_selftest_wait_timeout(_stream(stream)))


def check_device_status(stream=None):
    """Synchronise the stream and raise if a kernel's bounded wait gave up."""
    _check("ssm_check_device_status", load_library().ssm_check_device_status(_stream(stream)))


# ------------------------------------------------------------------ conv1d

def conv1d_fwd(x, w, bias, state0=None, *, out=None, state_last=None, want_state=True, stream=None):
    """Causal depthwise conv1d + SiLU.  x [B,L,D] (bf16/f32), w [D,K] f32, bias [D] f32,
    state0 [B,D,K-1] (act dtype, nullable).  Returns ``(out, state_last)``."""
    B, L, D = x.shape
    K = w.shape[1]
    if out is None:
        out = torch.empty_like(x)
    if want_state and state_last is None:
        state_last = torch.empty((B, D, K - 1), dtype=x.dtype, device=x.device)
    rc = load_library().ssm_conv1d_fwd(B, L, D, K, _act(x), _p(x), _p(w), _p(bias), _p(state0), _p(out),
                                       _p(state_last), _stream(stream))
    _check("ssm_conv1d_fwd", rc)
    return out, state_last


def conv1d_bwd_workspace_bytes(batch, seqlen, dim, width, act) -> int:
    return int(load_library().ssm_conv1d_bwd_workspace_bytes(batch, seqlen, dim, width, act))


def conv1d_bwd(x, w, bias, state0, dout, *, dx=None, want_dstate0=True, ws=None, stream=None):
    """Backward of ``sum(dout * out)``: dict dx (act dtype), dw, dbias, dstate0 (f32)."""
    B, L, D = x.shape
    K = w.shape[1]
    g = {"dx": torch.empty_like(x) if dx is None else dx, "dw": torch.empty_like(w), "dbias": torch.empty_like(bias),
         "dstate0": torch.empty((B, D, K - 1), dtype=torch.float32, device=x.device) if want_dstate0 else None}
    ws, wsb = _workspace(conv1d_bwd_workspace_bytes(B, L, D, K, _act(x)), x.device, ws)
    rc = load_library().ssm_conv1d_bwd(B, L, D, K, _act(x), _p(x), _p(w), _p(bias), _p(state0), _p(dout),
                                       _p(g["dx"]), _p(g["dw"]), _p(g["dbias"]), _p(g["dstate0"]), _p(ws),
                                       wsb, _stream(stream))
    _check("ssm_conv1d_bwd", rc)
    return g


def conv1d_step(x, w, bias, state, *, out=None, stream=None):
    """One step: x [B,D]; ``state`` [B,D,K-1] is shifted in place.  Returns ``out`` [B,D]."""
    B, D = x.shape
    K = w.shape[1]
    if out is None:
        out = torch.empty_like(x)
    rc = load_library().ssm_conv1d_step(B, D, K, _act(x), _p(x), _p(w), _p(bias), _p(state), _p(out),
                                        _stream(stream))
    _check("ssm_conv1d_step", rc)
    return out


def conv1d_path(x, w, dout=None, y=None):
    """Name of the kernel path ("tile", "vector" or "scalar") a conv1d call on
    these tensors takes; ``dout`` given asks about the backward (``y`` = dx),
    else the forward (``y`` = out).  A host-side query: nothing is launched."""
    B, L, D = x.shape
    K = w.shape[1]
    rc = load_library().ssm_conv1d_path(B, L, D, K, _act(x), _p(x), _p(dout), _p(y if y is not None else x))
    if rc < 0:
        _check("ssm_conv1d_path", -rc)
    return CONV_PATHS[rc]


SSD_CHUNK_LEN = 64


def ssd_fwd(x, dt_raw, dt_bias, A_log, Bm, Cm, Dp, h0=None, *, y=None, h_last=None, want_h_last=True,
            dt_limit=None, stream=None, save=False, chunk_states=None):
    """Mamba-2 SSD forward.  x [B,L,H,P], dt_raw [B,L,H], Bm/Cm [B,L,G,N] (bf16);
    dt_bias, A_log, Dp [H] f32; h0 [B,H,N,P] f32 (zeros when None).  Returns
    ``(y [B,L,H,P], h_last [B,H,N,P] or None)``, and with ``save`` also the
    chunk states ``[B,H,ceil(L/64),N,P]`` (bf16) that ssd_bwd reads."""
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    if y is None:
        y = torch.empty_like(x)
    if h_last is None and want_h_last:
        h_last = torch.empty((B, H, N, P), dtype=torch.float32, device=x.device)
    opts = _opts(dt_limit) if dt_limit is not None else None
    if not save:
        rc = load_library().ssm_ssd_fwd(B, L, H, P, G, N, _act(x), _p(x), _p(dt_raw), _p(dt_bias), _p(A_log),
                                        _p(Bm), _p(Cm), _p(Dp), _p(h0), _p(y), _p(h_last), opts, _stream(stream))
        _check("ssm_ssd_fwd", rc)
        return y, h_last
    nch = -(-L // SSD_CHUNK_LEN)
    if chunk_states is None:
        chunk_states = torch.empty((B, H, nch, N, P), dtype=torch.bfloat16, device=x.device)
    rc = load_library().ssm_ssd_fwd_save(B, L, H, P, G, N, _act(x), _p(x), _p(dt_raw), _p(dt_bias), _p(A_log),
                                         _p(Bm), _p(Cm), _p(Dp), _p(h0), _p(y), _p(h_last), _p(chunk_states),
                                         opts, _stream(stream))
    _check("ssm_ssd_fwd_save", rc)
    return y, h_last, chunk_states


def ssd_bwd_workspace_bytes(B, L, H, P, G, N, act=None) -> int:
    return int(load_library().ssm_ssd_bwd_workspace_bytes(B, L, H, P, G, N, SSM_BF16 if act is None else act))


def ssd_bwd(x, dt_raw, dt_bias, A_log, Bm, Cm, Dp, chunk_states, dy, dh_last=None, *, want_dh0=True,
            dt_limit=None, ws=None, grads=None, stream=None):
    """Mamba-2 SSD backward of ``sum(dy*y) + sum(dh_last*h_last)``.  Returns a
    dict: dx [B,L,H,P], ddt_raw [B,L,H], dBm/dCm [B,L,G,N] (bf16), ddt_bias,
    dA_log, dDp [H] (f32), dh0 [B,H,N,P] f32 (None unless ``want_dh0``)."""
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    dev = x.device
    g = dict(grads or {})
    g.setdefault("dx", torch.empty_like(x))
    g.setdefault("ddt_raw", torch.empty_like(dt_raw))
    g.setdefault("dBm", torch.empty_like(Bm))
    g.setdefault("dCm", torch.empty_like(Cm))
    g.setdefault("ddt_bias", torch.empty((H,), dtype=torch.float32, device=dev))
    g.setdefault("dA_log", torch.empty((H,), dtype=torch.float32, device=dev))
    g.setdefault("dDp", torch.empty((H,), dtype=torch.float32, device=dev))
    g.setdefault("dh0", torch.empty((B, H, N, P), dtype=torch.float32, device=dev) if want_dh0 else None)
    need = ssd_bwd_workspace_bytes(B, L, H, P, G, N, _act(x))
    if need < 0:
        raise SSMError("ssm_ssd_bwd_workspace_bytes", "SSM_ERR_UNSUPPORTED", f"shape {(B, L, H, P, G, N)}")
    ws, ws_bytes = _workspace(need, dev, ws)
    opts = _opts(dt_limit) if dt_limit is not None else None
    rc = load_library().ssm_ssd_bwd(B, L, H, P, G, N, _act(x), _p(x), _p(dt_raw), _p(dt_bias), _p(A_log), _p(Bm),
                                    _p(Cm), _p(Dp), _p(chunk_states), _p(dy), _p(dh_last), _p(g["dx"]),
                                    _p(g["ddt_raw"]), _p(g["ddt_bias"]), _p(g["dA_log"]), _p(g["dBm"]),
                                    _p(g["dCm"]), _p(g["dDp"]), _p(g["dh0"]), _p(ws), ws_bytes, opts,
                                    _stream(stream))
    _check("ssm_ssd_bwd", rc)
    return g
