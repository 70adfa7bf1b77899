"""fp64 CPU oracle of the Mamba-2 (SSD) mixer core -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports,
links or calls it, and the two share no code: this wrapper only marshals
numpy arrays into the plain C functions of ``ssd_oracle.c``.

Functions (each cites the passage it follows in ``ssd_oracle.c``):

* :func:`conv1d` -- causal depthwise conv over [conv state ; rows] with SiLU
  (TensorSharp "nemotron.md" sections 3 and 10; TensorRT-Model-Connect #2207
  "Implementation", add_short_conv_rows).
* :func:`ssd_sequential` -- the recurrence one row at a time (TensorSharp
  "nemotron.md" section 4.1).  This is the definition the GPU is held to.
* :func:`ssd_chunked` -- the chunk form for any partition of the rows
  (TensorRT-Model-Connect #2207 "Implementation"), brute force, used only to
  pin :func:`ssd_sequential`.
* :func:`decode_step` -- gather / one step / scatter at state slots (vllm.cpp
  #1362 summary; TensorSharp "nemotron.md" section 11).
* :func:`mixer_prefill` / :func:`mixer_decode` -- the compositions that the
  C-ABI calls ``ssd_chunk_scan`` / ``ssd_decode_step`` compute;
  :func:`mixer_prefill_varlen` -- ``ssd_chunk_scan_varlen``: packed sequences
  with their states at pool slots (vllm.cpp #1362 summary; TensorSharp
  "nemotron.md" section 11).
* :func:`gated_group_rmsnorm` -- group RMSNorm of y, then the SiLU(z) gate
  (TensorSharp "nemotron.md" sections 3, 4.1 and 6).
* :func:`segment_decay` / :func:`state_combine` -- a segment's total decay
  (the last element of its cumulative sum of dt A) and the state after two
  consecutive segments (TensorRT-Model-Connect #2207 "Implementation": the
  chunk form's carry, with a whole segment as the chunk); the pieces of
  sequence-parallel state passing.

Parity unpinned: none (see tests/test_oracle.py for the pins).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssd_oracle.so")

DT_SOFTPLUS = 1
HAS_Z = 2

_lib = None
_lock = threading.Lock()


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups")]


def build(force: bool = False, out_path: str | None = None, mutant: int = 0) -> str:
    """Compile ssd_oracle.c into a shared library (plain gcc, no fast-math).

    ``mutant`` != 0 builds a copy with one planted mistake (mutation tests
    only); it is always written to ``out_path``, never to the default path."""
    path = out_path or _LIB_PATH
    if mutant:
        assert out_path is not None and out_path != _LIB_PATH
    if force or mutant or not os.path.exists(path) or \
            os.path.getmtime(path) < os.path.getmtime(_SRC):
        tmp = path + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-fno-fast-math", f"-DORACLE_MUTANT={int(mutant)}",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, path)
    return path


def open_library(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_conv1d.restype = None
    lib.oracle_conv1d.argtypes = [ctypes.c_int] * 4 + [dp] * 6 + [ctypes.c_int]
    for name in ("oracle_ssd_sequential", "oracle_ssd_chunked"):
        getattr(lib, name).restype = ctypes.c_int
    lib.oracle_decode_step.restype = ctypes.c_int
    lib.oracle_segment_decay.restype = None
    lib.oracle_segment_decay.argtypes = [ctypes.c_int] * 3 + [ctypes.c_uint] + [dp] * 4
    lib.oracle_state_combine.restype = None
    lib.oracle_state_combine.argtypes = [ctypes.c_int, ctypes.c_long] + [dp] * 4
    lib.oracle_gated_group_rmsnorm.restype = None
    lib.oracle_gated_group_rmsnorm.argtypes = [ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_double] + [dp] * 4
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


def _dp(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def conv1d(xbc, conv_w, conv_b=None, state_in=None, apply_silu=True):
    """Causal depthwise conv (+SiLU).  xbc [B,S,C], conv_w [C,W], conv_b [C],
    state_in [B,W-1,C] or None (zeros).  Returns (out [B,S,C], state_out)."""
    xbc = _f64(xbc)
    conv_w = _f64(conv_w)
    conv_b = _f64(conv_b)
    state_in = _f64(state_in)
    B, S, C = xbc.shape
    W = conv_w.shape[1]
    assert conv_w.shape == (C, W)
    out = np.empty((B, S, C), np.float64)
    state_out = np.empty((B, W - 1, C), np.float64)
    _load().oracle_conv1d(B, S, C, W, _dp(xbc), _dp(conv_w), _dp(conv_b), _dp(state_in),
                          _dp(out), _dp(state_out), 1 if apply_silu else 0)
    return out, state_out


def _scan_common(xbc, dt_raw, dt_bias, A, D, z, h0, H, P, N, G):
    xbc = _f64(xbc)
    B, S, C = xbc.shape
    assert C == H * P + 2 * G * N, (C, H, P, G, N)
    dt_raw = _f64(dt_raw)
    assert dt_raw.shape == (B, S, H)
    arrs = dict(xbc=xbc, dt_raw=dt_raw, dt_bias=_f64(dt_bias), A=_f64(A), D=_f64(D),
                z=_f64(z), h0=_f64(h0))
    if arrs["z"] is not None:
        assert arrs["z"].shape == (B, S, H * P)
    if arrs["h0"] is not None:
        assert arrs["h0"].shape == (B, H, P, N)
    y = np.empty((B, S, H, P), np.float64)
    hS = np.empty((B, H, P, N), np.float64)
    dims = _Dims(B, S, H, P, N, G)
    return arrs, y, hS, dims


def ssd_sequential(xbc, dt_raw, A, *, H, P, N, G, dt_bias=None, D=None, z=None,
                   h0=None, dt_softplus=True, nthreads=None):
    """The recurrence over post-conv xbc [B,S,H*P+2*G*N].  Returns (y, hS)."""
    arrs, y, hS, dims = _scan_common(xbc, dt_raw, dt_bias, A, D, z, h0, H, P, N, G)
    flags = (DT_SOFTPLUS if dt_softplus else 0) | (HAS_Z if z is not None else 0)
    rc = _load().oracle_ssd_sequential(
        ctypes.byref(dims), ctypes.c_uint(flags), _dp(arrs["xbc"]), _dp(arrs["dt_raw"]),
        _dp(arrs["dt_bias"]), _dp(arrs["A"]), _dp(arrs["D"]), _dp(arrs["z"]),
        _dp(arrs["h0"]), _dp(y), _dp(hS), ctypes.c_int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_ssd_sequential rejected its arguments")
    return y, hS


def ssd_chunked(xbc, dt_raw, A, chunk_lens, *, H, P, N, G, dt_bias=None, D=None, z=None,
                h0=None, dt_softplus=True, nthreads=None):
    """The brute-force chunk form for the partition ``chunk_lens`` of S."""
    arrs, y, hS, dims = _scan_common(xbc, dt_raw, dt_bias, A, D, z, h0, H, P, N, G)
    lens = (ctypes.c_int * len(chunk_lens))(*[int(v) for v in chunk_lens])
    flags = (DT_SOFTPLUS if dt_softplus else 0) | (HAS_Z if z is not None else 0)
    rc = _load().oracle_ssd_chunked(
        ctypes.byref(dims), ctypes.c_uint(flags), _dp(arrs["xbc"]), _dp(arrs["dt_raw"]),
        _dp(arrs["dt_bias"]), _dp(arrs["A"]), _dp(arrs["D"]), _dp(arrs["z"]),
        _dp(arrs["h0"]), _dp(y), _dp(hS), lens, ctypes.c_int(len(chunk_lens)),
        ctypes.c_int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_ssd_chunked rejected its arguments")
    return y, hS


def decode_step(xbc, dt_raw, A, slot_ids, pool, *, H, P, N, G, dt_bias=None, D=None,
                z=None, dt_softplus=True):
    """One decode step at state slots.  xbc [R,Cdim] post-conv, dt_raw [R,H],
    pool [num_slots,H,P,N] (updated copy returned).  Returns (y [R,H,P], pool, rc)."""
    xbc = _f64(xbc)
    R = xbc.shape[0]
    dt_raw = _f64(dt_raw)
    pool = np.array(pool, dtype=np.float64, copy=True, order="C")
    slots = np.ascontiguousarray(np.asarray(slot_ids, dtype=np.int32))
    zz = _f64(z)
    y = np.zeros((R, H, P), np.float64)
    flags = (DT_SOFTPLUS if dt_softplus else 0) | (HAS_Z if zz is not None else 0)
    lib = _load()
    dtb, A_, D_ = _f64(dt_bias), _f64(A), _f64(D)
    rc = lib.oracle_decode_step(
        ctypes.c_int(R), ctypes.c_int(H), ctypes.c_int(P), ctypes.c_int(N), ctypes.c_int(G),
        ctypes.c_uint(flags), _dp(xbc), _dp(dt_raw), _dp(dtb), _dp(A_), _dp(D_), _dp(zz),
        slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), ctypes.c_int(pool.shape[0]),
        _dp(pool), _dp(y))
    return y, pool, rc


def mixer_prefill(xbc_raw, conv_w, dt_raw, A, *, H, P, N, G, conv_b=None, conv_state=None,
                  dt_bias=None, D=None, z=None, h0=None, dt_softplus=True, nthreads=None):
    """What one ssd_chunk_scan call computes: conv+SiLU over [conv state ; rows],
    then the recurrence.  conv_w=None means xbc_raw is already post-conv.
    Returns (y, hS, conv_state_out or None)."""
    if conv_w is not None:
        xbc, cs_out = conv1d(xbc_raw, conv_w, conv_b, conv_state, apply_silu=True)
    else:
        xbc, cs_out = _f64(xbc_raw), None
    y, hS = ssd_sequential(xbc, dt_raw, A, H=H, P=P, N=N, G=G, dt_bias=dt_bias, D=D, z=z,
                           h0=h0, dt_softplus=dt_softplus, nthreads=nthreads)
    return y, hS, cs_out


def mixer_prefill_varlen(xbc_raw, conv_w, dt_raw, A, cu_seqlens, slot_ids, ssm_pool,
                         conv_pool, *, H, P, N, G, has_initial_state=None, conv_b=None,
                         dt_bias=None, D=None, z=None, dt_softplus=True, nthreads=None):
    """What one ssd_chunk_scan_varlen call computes: sequences packed row after
    row (sequence i = rows cu_seqlens[i] .. cu_seqlens[i+1]-1), each run as one
    mixer_prefill from the states at its pool slot (zeros when
    has_initial_state[i] is 0: a fresh request), the final states written back
    at the slot (vllm.cpp #1362 summary: the prefill half of a mixed batch over
    packed rows, states at the state index; TensorSharp "nemotron.md" section
    11: per-slot state pools).  xbc_raw [T,Cdim], dt_raw [T,H], z [T,H*P] or
    None, pools [slots,...].  Returns (y [T,H,P], ssm_pool', conv_pool')."""
    xbc_raw = _f64(xbc_raw)
    dt_raw = _f64(dt_raw)
    z = _f64(z)
    ssm_pool = np.array(ssm_pool, dtype=np.float64, copy=True)
    conv_pool = None if conv_pool is None else np.array(conv_pool, dtype=np.float64, copy=True)
    T = xbc_raw.shape[0]
    y = np.zeros((T, H, P), np.float64)
    for i in range(len(slot_ids)):
        r0, r1, sl = int(cu_seqlens[i]), int(cu_seqlens[i + 1]), int(slot_ids[i])
        init = has_initial_state is None or bool(has_initial_state[i])
        h0 = ssm_pool[sl][None] if init else None
        cs = conv_pool[sl][None] if (init and conv_pool is not None) else None
        yi, hS, cs_out = mixer_prefill(
            xbc_raw[None, r0:r1], conv_w, dt_raw[None, r0:r1], A, H=H, P=P, N=N, G=G,
            conv_b=conv_b, conv_state=cs, dt_bias=dt_bias, D=D,
            z=None if z is None else z[None, r0:r1], h0=h0, dt_softplus=dt_softplus,
            nthreads=nthreads)
        y[r0:r1] = yi[0]
        ssm_pool[sl] = hS[0]
        if conv_pool is not None and cs_out is not None:
            conv_pool[sl] = cs_out[0]
    return y, ssm_pool, conv_pool


def mixer_decode(xbc_raw, conv_w, dt_raw, A, slot_ids, ssm_pool, *, H, P, N, G,
                 conv_b=None, conv_pool=None, dt_bias=None, D=None, z=None,
                 dt_softplus=True):
    """What one ssd_decode_step call computes: for each row, the conv over the
    slot's conv state plus the new row (conv pool rolled by one row), then one
    recurrence step at the slot.  Returns (y, ssm_pool, conv_pool or None)."""
    slots = np.asarray(slot_ids, dtype=np.int64)
    if conv_w is not None:
        cp = np.array(conv_pool, dtype=np.float64, copy=True)
        raw = _f64(xbc_raw)[:, None, :]
        st_in = cp[slots]
        xbc, st_out = conv1d(raw, conv_w, conv_b, st_in, apply_silu=True)
        xbc = xbc[:, 0, :]
        cp[slots] = st_out
    else:
        xbc, cp = _f64(xbc_raw), None
    y, pool, rc = decode_step(xbc, dt_raw, A, slot_ids, ssm_pool, H=H, P=P, N=N, G=G,
                              dt_bias=dt_bias, D=D, z=z, dt_softplus=dt_softplus)
    if rc != 0:
        raise ValueError("oracle decode: slot id out of range")
    return y, pool, cp


def gated_group_rmsnorm(y, z, w, eps, G):
    """out = silu(z) * y / sqrt(mean over the group of y^2 + eps) * w, with G
    groups of contiguous channels on the last axis (TensorSharp "nemotron.md"
    sections 3, 4.1, 6).  y, z [..., C]; w [C].  Returns out [..., C]."""
    y = _f64(y)
    z = _f64(z)
    w = _f64(w)
    C = y.shape[-1]
    assert z.shape == y.shape and w.shape == (C,) and C % G == 0
    out = np.empty_like(y)
    rows = y.size // C
    _load().oracle_gated_group_rmsnorm(rows, C, G, float(eps), _dp(y), _dp(z), _dp(w), _dp(out))
    return out



def segment_decay(dt_raw, A, *, dt_bias=None, dt_softplus=True):
    """gamma[b,h] = sum_t dt[b,t,h] * A[h] over the rows of dt_raw [B,S,H]."""
    dt_raw = _f64(dt_raw)
    B, S, H = dt_raw.shape
    A_ = _f64(A)
    dtb = _f64(dt_bias)
    out = np.empty((B, H), np.float64)
    _load().oracle_segment_decay(B, S, H, DT_SOFTPLUS if dt_softplus else 0, _dp(dt_raw),
                                 _dp(dtb), _dp(A_), _dp(out))
    return out


def state_combine(gamma, h_prev, h_seg):
    """exp(min(gamma, 0)) * h_prev + h_seg per (sequence, head); gamma [B,H],
    states [B,H,P,N]; h_prev None means zeros."""
    g = _f64(gamma)
    hs = _f64(h_seg)
    hp = _f64(h_prev)
    B, H = g.shape
    assert hs.shape[:2] == (B, H) and (hp is None or hp.shape == hs.shape)
    out = np.empty_like(hs)
    _load().oracle_state_combine(B * H, hs.shape[2] * hs.shape[3], _dp(g), _dp(hp), _dp(hs),
                                 _dp(out))
    return out
