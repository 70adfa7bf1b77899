"""Python binding of the GB300 SSD mixer-core library (``libssd_gb300.so``).

The functions below carry the names of the C-ABI entry points declared in
``include/ssd.h`` and only marshal arguments: torch tensors (device memory,
used for allocation and streams only) become raw pointers, ``None`` becomes
NULL, and a non-OK status raises :class:`SsdError`.  Every step of the
computation runs in the library's CUDA kernels; there is no other path.  If
the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssd_gb300.so")

SSD_OK = 0
SSD_ERR_INVALID_ARG = 1
SSD_ERR_UNSUPPORTED = 2
SSD_ERR_CUDA = 3
SSD_ERR_BAD_SLOT = 4
SSD_ERR_TIMEOUT = 5
SSD_ERR_DUPLICATE_SLOT = 6

SSD_CHECK_DISTINCT_SLOTS = 1

SSD_F32 = 0
SSD_BF16 = 1

SSD_DT_SOFTPLUS = 1
SSD_HAS_Z = 2
SSD_GATED_NORM = 4

# size of the fixed per-GPU scratch array behind ssd_chunk_scan_static_ws
SSD_STATIC_SCRATCH_BYTES = 16 << 20

# every symbol include/ssd.h declares
EXPORTED = ("ssd_conv1d_rows", "ssd_chunk_scan", "ssd_chunk_scan_workspace_size",
            "ssd_decode_step", "ssd_status_string", "ssd_read_device_error",
            "ssd_launch_counts", "ssd_chunk_scan_static_ws", "ssd_gated_group_rmsnorm",
            "ssd_chunk_scan_varlen", "ssd_set_debug_checks", "ssd_set_wait_limit_ns",
            "ssd_segment_decay", "ssd_state_combine", "ssd_chunk_scan_gated_norm")

KERNEL_KINDS = ("conv_rows", "conv_state", "scan_simt", "scan_tc", "bc_conv", "decode_step",
                "decode_conv", "gated_norm", "segment_decay", "state_combine", "norm_scale")


class SsdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {ssd_status_string(status)} (status {status})")


class ssd_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("batch", "seqlen", "nheads", "headdim", "dstate",
                                            "ngroups", "conv_width", "chunk")]

    @property
    def cdim(self) -> int:
        return self.nheads * self.headdim + 2 * self.ngroups * self.dstate


def dims(batch, seqlen, nheads, headdim, dstate, ngroups, conv_width=4, chunk=128) -> ssd_dims:
    return ssd_dims(batch, seqlen, nheads, headdim, dstate, ngroups, conv_width, chunk)


_lib = None
_lock = threading.Lock()
_vp = ctypes.c_void_p


def load_library():
    """Load libssd_gb300.so (raises if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m ssd_scan_gb300.build` "
                    "(nvcc, sm_103a); the SSD library has no CPU fallback")
            lib = ctypes.CDLL(LIB_PATH)
            P = ctypes.POINTER(ssd_dims)
            ci, cu, sz = ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
            lib.ssd_conv1d_rows.argtypes = [P, ci, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
            lib.ssd_chunk_scan.argtypes = [P, ci, cu] + [_vp] * 14 + [sz, _vp]
            lib.ssd_chunk_scan_static_ws.argtypes = [P, ci, cu] + [_vp] * 13 + [_vp]
            lib.ssd_chunk_scan_gated_norm.argtypes = [P, ci, cu] + [_vp] * 11 + \
                [ctypes.c_float] + [_vp] * 4 + [sz, _vp]
            lib.ssd_chunk_scan_workspace_size.argtypes = [P, ci, cu, ci, ctypes.POINTER(sz)]
            lib.ssd_decode_step.argtypes = [P, ci, cu] + [_vp] * 10 + [ci, _vp, _vp, _vp]
            lib.ssd_gated_group_rmsnorm.argtypes = [P, ci, _vp, _vp, _vp, ctypes.c_float, _vp,
                                                     _vp]
            lib.ssd_chunk_scan_varlen.argtypes = [P, ci, cu, _vp, _vp, _vp, ci] + [_vp] * 11 + \
                [_vp, sz, _vp]
            lib.ssd_status_string.argtypes = [ci]
            lib.ssd_status_string.restype = ctypes.c_char_p
            lib.ssd_read_device_error.argtypes = [_vp]
            lib.ssd_launch_counts.argtypes = [ctypes.POINTER(ctypes.c_uint64), ci]
            lib.ssd_segment_decay.argtypes = [P, cu, _vp, _vp, _vp, _vp, _vp]
            lib.ssd_state_combine.argtypes = [P, _vp, _vp, _vp, _vp, _vp]
            lib.ssd_set_debug_checks.argtypes = [cu]
            lib.ssd_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            for n in EXPORTED:
                if n != "ssd_status_string":
                    getattr(lib, n).restype = ci
            lib.ssd_set_debug_checks.restype = cu
            lib.ssd_set_wait_limit_ns.restype = ctypes.c_uint64
            _lib = lib
    return _lib


def ssd_set_debug_checks(flags: int) -> int:
    """Process-wide debug checks (SSD_CHECK_DISTINCT_SLOTS); returns the old flags."""
    return int(load_library().ssd_set_debug_checks(int(flags)))


def ssd_set_wait_limit_ns(ns: int) -> int:
    """Bound on each wait inside the tensor-core scan kernel (0: the default
    2 s); returns the old bound."""
    return int(load_library().ssd_set_wait_limit_ns(int(ns)))


def ssd_segment_decay(d: ssd_dims, flags: int, dt, dt_bias, A, gamma, stream=None) -> None:
    f = torch.float32
    _check(load_library().ssd_segment_decay(
        ctypes.byref(d), flags, _ptr(dt, f, "dt"), _ptr(dt_bias, f, "dt_bias"), _ptr(A, f, "A"),
        _ptr(gamma, f, "gamma"), _stream(stream)), "ssd_segment_decay")


def ssd_state_combine(d: ssd_dims, gamma, h_prev, h_seg, h_out, stream=None) -> None:
    f = torch.float32
    _check(load_library().ssd_state_combine(
        ctypes.byref(d), _ptr(gamma, f, "gamma"), _ptr(h_prev, f, "h_prev"),
        _ptr(h_seg, f, "h_seg"), _ptr(h_out, f, "h_out"), _stream(stream)), "ssd_state_combine")


def ssd_status_string(status: int) -> str:
    return load_library().ssd_status_string(int(status)).decode()


_ACT = {SSD_F32: torch.float32, SSD_BF16: torch.bfloat16}


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor or None")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA (device) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return _vp(t.data_ptr())


def _stream(stream):
    if stream is None:
        return _vp(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return _vp(stream.cuda_stream)
    return _vp(int(stream))


def _check(status, where):
    if status != SSD_OK:
        raise SsdError(status, where)


def act_of(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SSD_BF16
    if t.dtype == torch.float32:
        return SSD_F32
    raise TypeError(f"unsupported activation dtype {t.dtype}")


def ssd_conv1d_rows(d: ssd_dims, act: int, xbc_in, conv_w, conv_b, conv_state_in, xbc_out,
                    conv_state_out, stream=None) -> None:
    a = _ACT[act]
    f = torch.float32
    _check(load_library().ssd_conv1d_rows(
        ctypes.byref(d), act, _ptr(xbc_in, a, "xbc_in"), _ptr(conv_w, f, "conv_w"),
        _ptr(conv_b, f, "conv_b"), _ptr(conv_state_in, a, "conv_state_in"),
        _ptr(xbc_out, a, "xbc_out"), _ptr(conv_state_out, a, "conv_state_out"),
        _stream(stream)), "ssd_conv1d_rows")


def ssd_chunk_scan_workspace_size(d: ssd_dims, act: int, flags: int, conv_fused: bool) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().ssd_chunk_scan_workspace_size(ctypes.byref(d), act, flags,
                                                         1 if conv_fused else 0,
                                                         ctypes.byref(out)),
           "ssd_chunk_scan_workspace_size")
    return int(out.value)


def ssd_chunk_scan(d: ssd_dims, act: int, flags: int, xbc, conv_w, conv_b, conv_state_in,
                   conv_state_out, dt, dt_bias, A, D, z, ssm_state_in, y, ssm_state_out,
                   workspace=None, stream=None) -> None:
    a = _ACT[act]
    f = torch.float32
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().ssd_chunk_scan(
        ctypes.byref(d), act, flags, _ptr(xbc, a, "xbc"), _ptr(conv_w, f, "conv_w"),
        _ptr(conv_b, f, "conv_b"), _ptr(conv_state_in, a, "conv_state_in"),
        _ptr(conv_state_out, a, "conv_state_out"), _ptr(dt, f, "dt"),
        _ptr(dt_bias, f, "dt_bias"), _ptr(A, f, "A"), _ptr(D, f, "D"), _ptr(z, a, "z"),
        _ptr(ssm_state_in, f, "ssm_state_in"), _ptr(y, a, "y"),
        _ptr(ssm_state_out, f, "ssm_state_out"), _ptr(workspace, None, "workspace"),
        ws_bytes, _stream(stream)), "ssd_chunk_scan")


def ssd_chunk_scan_gated_norm(d: ssd_dims, act: int, flags: int, xbc, conv_w, conv_b,
                              conv_state_in, conv_state_out, dt, dt_bias, A, D, z, norm_w,
                              eps: float, ssm_state_in, y, ssm_state_out, workspace=None,
                              stream=None) -> None:
    """The scan, then silu(z) * GroupRMSNorm(y; norm_w, eps) over its output,
    in one call (workspace: ssd_chunk_scan_workspace_size with SSD_GATED_NORM)."""
    a = _ACT[act]
    f = torch.float32
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().ssd_chunk_scan_gated_norm(
        ctypes.byref(d), act, flags, _ptr(xbc, a, "xbc"), _ptr(conv_w, f, "conv_w"),
        _ptr(conv_b, f, "conv_b"), _ptr(conv_state_in, a, "conv_state_in"),
        _ptr(conv_state_out, a, "conv_state_out"), _ptr(dt, f, "dt"),
        _ptr(dt_bias, f, "dt_bias"), _ptr(A, f, "A"), _ptr(D, f, "D"), _ptr(z, a, "z"),
        _ptr(norm_w, f, "norm_w"), ctypes.c_float(eps), _ptr(ssm_state_in, f, "ssm_state_in"),
        _ptr(y, a, "y"), _ptr(ssm_state_out, f, "ssm_state_out"),
        _ptr(workspace, None, "workspace"), ws_bytes, _stream(stream)),
        "ssd_chunk_scan_gated_norm")


def ssd_chunk_scan_static_ws(d: ssd_dims, act: int, flags: int, xbc, conv_w, conv_b,
                             conv_state_in, conv_state_out, dt, dt_bias, A, D, z, ssm_state_in,
                             y, ssm_state_out, stream=None) -> None:
    """ssd_chunk_scan without a workspace argument, for callers that cannot
    allocate device memory: the scratch is the library's fixed per-GPU array
    (SSD_STATIC_SCRATCH_BYTES); calls that overlap on one GPU race on it."""
    a = _ACT[act]
    f = torch.float32
    _check(load_library().ssd_chunk_scan_static_ws(
        ctypes.byref(d), act, flags, _ptr(xbc, a, "xbc"), _ptr(conv_w, f, "conv_w"),
        _ptr(conv_b, f, "conv_b"), _ptr(conv_state_in, a, "conv_state_in"),
        _ptr(conv_state_out, a, "conv_state_out"), _ptr(dt, f, "dt"),
        _ptr(dt_bias, f, "dt_bias"), _ptr(A, f, "A"), _ptr(D, f, "D"), _ptr(z, a, "z"),
        _ptr(ssm_state_in, f, "ssm_state_in"), _ptr(y, a, "y"),
        _ptr(ssm_state_out, f, "ssm_state_out"), _stream(stream)), "ssd_chunk_scan_static_ws")


def ssd_decode_step(d: ssd_dims, act: int, flags: int, xbc, conv_w, conv_b, conv_pool, dt,
                    dt_bias, A, D, z, slot_ids, num_slots: int, ssm_pool, y,
                    stream=None) -> None:
    a = _ACT[act]
    f = torch.float32
    _check(load_library().ssd_decode_step(
        ctypes.byref(d), act, flags, _ptr(xbc, a, "xbc"), _ptr(conv_w, f, "conv_w"),
        _ptr(conv_b, f, "conv_b"), _ptr(conv_pool, a, "conv_pool"), _ptr(dt, f, "dt"),
        _ptr(dt_bias, f, "dt_bias"), _ptr(A, f, "A"), _ptr(D, f, "D"), _ptr(z, a, "z"),
        _ptr(slot_ids, torch.int32, "slot_ids"), int(num_slots),
        _ptr(ssm_pool, f, "ssm_pool"), _ptr(y, a, "y"), _stream(stream)), "ssd_decode_step")


def ssd_chunk_scan_varlen(d: ssd_dims, act: int, flags: int, cu_seqlens, slot_ids,
                          has_initial_state, num_slots: int, xbc, conv_w, conv_b, conv_pool, dt,
                          dt_bias, A, D, z, ssm_pool, y, workspace=None, stream=None) -> None:
    """The scan over packed sequences (d.batch sequences, d.seqlen rows in all),
    states at pool slots, updated in place."""
    a = _ACT[act]
    f = torch.float32
    i32 = torch.int32
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().ssd_chunk_scan_varlen(
        ctypes.byref(d), act, flags, _ptr(cu_seqlens, i32, "cu_seqlens"),
        _ptr(slot_ids, i32, "slot_ids"), _ptr(has_initial_state, i32, "has_initial_state"),
        int(num_slots), _ptr(xbc, a, "xbc"), _ptr(conv_w, f, "conv_w"), _ptr(conv_b, f, "conv_b"),
        _ptr(conv_pool, a, "conv_pool"), _ptr(dt, f, "dt"), _ptr(dt_bias, f, "dt_bias"),
        _ptr(A, f, "A"), _ptr(D, f, "D"), _ptr(z, a, "z"), _ptr(ssm_pool, f, "ssm_pool"),
        _ptr(y, a, "y"), _ptr(workspace, None, "workspace"), ws_bytes, _stream(stream)),
        "ssd_chunk_scan_varlen")


def ssd_gated_group_rmsnorm(d: ssd_dims, act: int, y, z, weight, eps: float, out,
                            stream=None) -> None:
    """out = silu(z) * GroupRMSNorm(y; weight, eps), d.ngroups groups of the
    H*P channels of each row; out may be y itself."""
    a = _ACT[act]
    _check(load_library().ssd_gated_group_rmsnorm(
        ctypes.byref(d), act, _ptr(y, a, "y"), _ptr(z, a, "z"),
        _ptr(weight, torch.float32, "weight"), ctypes.c_float(eps), _ptr(out, a, "out"),
        _stream(stream)), "ssd_gated_group_rmsnorm")


def ssd_launch_counts() -> dict:
    """Process-wide number of kernels the library launched, per kernel kind."""
    buf = (ctypes.c_uint64 * len(KERNEL_KINDS))()
    n = load_library().ssd_launch_counts(buf, len(KERNEL_KINDS))
    assert n == len(KERNEL_KINDS), n
    return {k: int(buf[i]) for i, k in enumerate(KERNEL_KINDS)}


def ssd_read_device_error(stream=None) -> int:
    """Synchronise the stream; return and clear the device error word (a status)."""
    return int(load_library().ssd_read_device_error(_stream(stream)))


# ---------------------------------------------------------------------------
# allocation helpers (torch allocates; the library computes)

def workspace_for(d: ssd_dims, act: int, flags: int, conv_fused: bool, device) -> torch.Tensor | None:
    n = ssd_chunk_scan_workspace_size(d, act, flags, conv_fused)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device)


def chunk_scan(xbc, dt, A, *, nheads, headdim, dstate, ngroups, conv_w=None, conv_b=None,
               conv_state=None, dt_bias=None, D=None, z=None, ssm_state=None,
               dt_softplus=True, out=None, workspace=None, stream=None, norm_w=None,
               norm_eps=1e-5):
    """Allocate outputs and call ssd_chunk_scan (with ``norm_w``:
    ssd_chunk_scan_gated_norm, z required).  Returns (y, ssm_state_out,
    conv_state_out or None)."""
    B, S, _ = xbc.shape
    W = conv_w.shape[1] if conv_w is not None else 4
    d = dims(B, S, nheads, headdim, dstate, ngroups, W, 128)
    act = act_of(xbc)
    flags = (SSD_DT_SOFTPLUS if dt_softplus else 0) | (SSD_HAS_Z if z is not None else 0)
    if norm_w is not None:
        if z is None:
            raise ValueError("the gated norm needs z")
        flags = (flags & SSD_DT_SOFTPLUS) | SSD_GATED_NORM
    if out is None:
        y = torch.empty((B, S, nheads, headdim), dtype=xbc.dtype, device=xbc.device)
        hs = torch.empty((B, nheads, headdim, dstate), dtype=torch.float32, device=xbc.device)
        cs = (torch.empty((B, W - 1, d.cdim), dtype=xbc.dtype, device=xbc.device)
              if conv_w is not None else None)
    else:
        y, hs, cs = out
    if workspace is None:
        workspace = workspace_for(d, act, flags, conv_w is not None, xbc.device)
    if norm_w is not None:
        ssd_chunk_scan_gated_norm(d, act, flags, xbc, conv_w, conv_b, conv_state, cs, dt,
                                  dt_bias, A, D, z, norm_w, norm_eps, ssm_state, y, hs,
                                  workspace, stream)
    else:
        ssd_chunk_scan(d, act, flags, xbc, conv_w, conv_b, conv_state, cs, dt, dt_bias, A, D,
                       z, ssm_state, y, hs, workspace, stream)
    return y, hs, cs


def gated_group_rmsnorm(y, z, weight, *, ngroups, eps=1e-5, out=None, stream=None):
    """Group RMSNorm of y [B,S,H,P] (or [B,S,H*P]) then the SiLU(z) gate, z
    [B,S,H*P]; returns out shaped like y (a new tensor unless ``out`` is given,
    which may be y itself)."""
    B, S = y.shape[0], y.shape[1]
    C = weight.numel()
    if C % ngroups:
        raise ValueError(f"{C} channels do not split into {ngroups} groups")
    d = dims(B, S, ngroups, C // ngroups, 1, ngroups)  # channels as ngroups heads of C/ngroups
    o = torch.empty_like(y) if out is None else out
    ssd_gated_group_rmsnorm(d, act_of(y), y, z, weight, eps, o, stream)
    return o

