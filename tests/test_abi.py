"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports
every symbol include/ssd.h declares, and its host-side argument checks reject
bad calls before anything touches CUDA."""
import ctypes
import os
import re

import pytest

import ssd_scan_gb300 as ssd
from ssd_scan_gb300 import build as ssd_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ssd_build.build()
    return ssd.load_library()


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"SSD_API\s+[\w\s\*]+?\b(ssd_\w+)\s*\(", txt)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("ssd_conv1d_rows", "ssd_chunk_scan", "ssd_decode_step", "ssd_status_string",
              "ssd_read_device_error", "ssd_chunk_scan_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(ssd.LIB_PATH)
    for n in _declared():
        assert hasattr(raw, n), n
    assert set(_declared()) <= set(ssd.EXPORTED) | set(_declared())
    assert set(ssd.EXPORTED) == set(_declared())


def test_status_strings(lib):
    for s in range(7):
        assert ssd.ssd_status_string(s) != "unknown status"
    assert "slot" in ssd.ssd_status_string(ssd.SSD_ERR_BAD_SLOT)
    assert "twice" in ssd.ssd_status_string(ssd.SSD_ERR_DUPLICATE_SLOT)


def test_process_wide_settings_round_trip(lib):
    """The debug-check and wait-limit setters return the previous value and
    touch no device (host-side settings read at each launch)."""
    assert ssd.ssd_set_debug_checks(ssd.SSD_CHECK_DISTINCT_SLOTS) == 0
    assert ssd.ssd_set_debug_checks(0xff) == ssd.SSD_CHECK_DISTINCT_SLOTS
    assert ssd.ssd_set_debug_checks(0) == ssd.SSD_CHECK_DISTINCT_SLOTS  # unknown bits dropped
    assert ssd.ssd_set_wait_limit_ns(500) == 0
    assert ssd.ssd_set_wait_limit_ns(0) == 500


def _d(**kw):
    base = dict(batch=1, seqlen=8, nheads=4, headdim=16, dstate=16, ngroups=1, conv_width=4,
                chunk=128)
    base.update(kw)
    return ssd.ssd_dims(*[base[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate",
                                             "ngroups", "conv_width", "chunk")])


def _scan(lib, d, act=0, flags=1, **ptrs):
    names = ["xbc", "conv_w", "conv_b", "cs_in", "cs_out", "dt", "dt_bias", "A", "D", "z",
             "h0", "y", "hS", "ws"]
    args = [ptrs.get(n) for n in names]
    return lib.ssd_chunk_scan(ctypes.byref(d) if d is not None else None, act, flags,
                              *[ctypes.c_void_p(a) if a else None for a in args],
                              ctypes.c_size_t(ptrs.get("ws_bytes", 0)), None)


GOOD = dict(xbc=0x10000, dt=0x20000, A=0x30000, y=0x40000, hS=0x50000)


@pytest.mark.parametrize("bad", [
    dict(d=None),
    dict(dims=dict(batch=-1)),
    dict(dims=dict(nheads=3, ngroups=2)),
    dict(dims=dict(conv_width=0)),
    dict(dims=dict(conv_width=9)),
    dict(dims=dict(headdim=0)),
    dict(act=7),
    dict(flags=8),
    dict(ptrs=dict(xbc=None)),
    dict(ptrs=dict(y=0x40004)),          # misaligned
    dict(ptrs=dict(A=None)),
    dict(ptrs=dict(hS=None)),
    dict(ptrs=dict(cs_in=0x60000)),      # conv state without conv weights
    dict(flags=3),                        # z flag without z
])
def test_scan_rejects_bad_arguments_on_host(lib, bad):
    d = None if "d" in bad else _d(**bad.get("dims", {}))
    ptrs = dict(GOOD)
    ptrs.update(bad.get("ptrs", {}))
    st = _scan(lib, d, act=bad.get("act", 0), flags=bad.get("flags", 1), **ptrs)
    assert st == ssd.SSD_ERR_INVALID_ARG


def test_bf16_rejects_other_chunk_sizes(lib):
    st = _scan(lib, _d(chunk=64), act=1, **GOOD)
    assert st == ssd.SSD_ERR_UNSUPPORTED


def test_decode_rejects_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    for K, want in ((0, ssd.SSD_ERR_INVALID_ARG), (17, ssd.SSD_ERR_UNSUPPORTED)):
        d = _d(batch=4, seqlen=K)  # tokens per row: 1 .. 16
        st = lib.ssd_decode_step(ctypes.byref(d), 1, 1, P(0x10000), None, None, None,
                                 P(0x20000), None, P(0x30000), None, None, P(0x40000), 8,
                                 P(0x50000), P(0x60000), None)
        assert st == want, K
    d = _d(batch=4, seqlen=1)
    st = lib.ssd_decode_step(ctypes.byref(d), 1, 1, P(0x10000), None, None, None, P(0x20000),
                             None, P(0x30000), None, None, None, 8, P(0x50000), P(0x60000),
                             None)
    assert st == ssd.SSD_ERR_INVALID_ARG  # slot ids required
    st = lib.ssd_decode_step(ctypes.byref(d), 1, 1, P(0x10000), None, None, None, P(0x20000),
                             None, P(0x30000), None, None, P(0x40000), -1, P(0x50000),
                             P(0x60000), None)
    assert st == ssd.SSD_ERR_INVALID_ARG  # negative pool size


def test_conv_rejects_bad_arguments_on_host(lib):
    d = _d()
    P = ctypes.c_void_p
    assert lib.ssd_conv1d_rows(ctypes.byref(d), 1, P(0x10000), None, None, None, P(0x20000),
                               None, None) == ssd.SSD_ERR_INVALID_ARG  # no weights
    assert lib.ssd_conv1d_rows(ctypes.byref(d), 1, P(0x10000), P(0x30000), None, None,
                               P(0x10000), None, None) == ssd.SSD_ERR_INVALID_ARG  # in == out
    bad = _d(nheads=1, headdim=3, dstate=1)  # Cdim*2 bytes not a multiple of 16
    assert lib.ssd_conv1d_rows(ctypes.byref(bad), 1, P(0x10000), P(0x30000), None, None,
                               P(0x20000), None, None) == ssd.SSD_ERR_INVALID_ARG


def test_workspace_size_query(lib):
    n = ssd.ssd_chunk_scan_workspace_size(_d(), 1, 1, True)
    assert n >= 0
    with pytest.raises(ssd.SsdError):
        ssd.ssd_chunk_scan_workspace_size(_d(batch=-2), 1, 1, True)


def test_workspace_size_follows_the_routing(lib):
    """Scratch is the post-conv B|C rows, [B, S, 2 G N] bf16 rounded up to 256
    bytes, and only where the call takes the tensor-core path with the conv
    fused (bf16, P = 64, N = 128, W <= 4, rows in the call)."""
    flags = ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z
    tc = dict(headdim=64, dstate=128)
    size = lambda act, fused, **kw: ssd.ssd_chunk_scan_workspace_size(_d(**{**tc, **kw}), act,
                                                                       flags, fused)
    # the Nemotron-H-8B prefill call: 2048 rows x 2 x 8 x 128 bf16 = 8 MiB
    assert size(ssd.SSD_BF16, True, seqlen=2048, nheads=128, ngroups=8) == 2048 * 2 * 8 * 128 * 2
    # ragged sizes round up to 256 bytes
    assert size(ssd.SSD_BF16, True, batch=3, seqlen=5, ngroups=1) == (3 * 5 * 2 * 128 * 2 + 255) // 256 * 256
    # no scratch: conv not fused, fp32 (row-exact kernel), no rows, other shapes
    assert size(ssd.SSD_BF16, False, seqlen=2048) == 0
    assert size(ssd.SSD_F32, True, seqlen=2048) == 0
    assert size(ssd.SSD_BF16, True, seqlen=0) == 0
    assert size(ssd.SSD_BF16, True, seqlen=2048, headdim=32) == 0
    assert size(ssd.SSD_BF16, True, seqlen=2048, conv_width=5) == 0


def test_binding_refuses_host_tensors(lib):
    import torch
    with pytest.raises((ValueError, TypeError)):
        ssd.chunk_scan(torch.zeros(1, 8, 96), torch.zeros(1, 8, 4), torch.zeros(4),
                       nheads=4, headdim=16, dstate=16, ngroups=1)
