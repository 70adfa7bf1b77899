"""Failure detection on the GPU without a fault: a bounded device wait that
runs out, and slot ids given twice, each reported through the device error
word while the context stays usable.

The time-out is made by shortening the bound on the scan kernel's waits
between its warps (ssd_set_wait_limit_ns) to 1 ns, so that the first wait not
already satisfied gives up: the kernel then stops early, waits (with its full
bound) for its own copies and tensor-core work in flight, frees its tensor
memory and reports SSD_ERR_TIMEOUT.  No trap, no bad address, no endless loop:
the next call with the default bound must match the oracle.
"""
import numpy as np
import pytest
import torch

import ssd_inputs as si
from tests.helpers import TOL, assert_close, gpu_prefill, make_problem, oracle_prefill

pytestmark = pytest.mark.gpu

ssd = pytest.importorskip("ssd_scan_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ssd.load_library()
    assert ssd.ssd_read_device_error() == ssd.SSD_OK
    yield
    ssd.ssd_set_wait_limit_ns(0)
    ssd.ssd_set_debug_checks(0)
    assert ssd.ssd_read_device_error() == ssd.SSD_OK


def test_bounded_wait_runs_out_then_next_call_is_correct():
    shape = si.Shape(batch=1, seqlen=512, nheads=4, headdim=64, dstate=128, ngroups=1)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=21)
    old = ssd.ssd_set_wait_limit_ns(1)
    try:
        gpu_prefill(shape, dev)
        assert ssd.ssd_read_device_error() == ssd.SSD_ERR_TIMEOUT
    finally:
        ssd.ssd_set_wait_limit_ns(old)
    assert ssd.ssd_read_device_error() == ssd.SSD_OK  # the read cleared it
    y, h, cs = gpu_prefill(shape, dev)
    assert ssd.ssd_read_device_error() == ssd.SSD_OK
    yo, ho, co, cols = oracle_prefill(shape, cpu)
    assert_close(y, yo, TOL[torch.bfloat16], what="y after a timed-out call")
    assert_close(h, ho, TOL[torch.bfloat16], what="state after a timed-out call")


def _decode_call(shape, prm, xbc, dt, z, slots, pool, cpool):
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    R = xbc.shape[0]
    y = torch.full((R, H, P), float("nan"), dtype=torch.bfloat16, device="cuda")
    ssd.ssd_decode_step(ssd.dims(R, 1, H, P, N, G, shape.conv_width), ssd.SSD_BF16,
                        ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z, xbc, prm["conv_w"], prm["conv_b"],
                        cpool, dt, prm["dt_bias"], prm["A"], prm["D"], z,
                        torch.tensor(slots, dtype=torch.int32, device="cuda"), pool.shape[0],
                        pool, y)
    return y


def test_duplicate_decode_slot_reported_and_skipped_with_debug_checks():
    """Rows at slots [2, 5, 2, 7] with the distinct-slot check on: the second
    row at slot 2 writes nothing and sets SSD_ERR_DUPLICATE_SLOT; the pools and
    the other rows' y are bit for bit those of the call without that row."""
    shape = si.Shape(batch=4, seqlen=1, nheads=8, headdim=64, dstate=128, ngroups=2)
    prm = {k: v.cuda() for k, v in si.params(shape, seed=2).items()}
    pools = si.decode_pools(shape, 8, seed=2, device="cuda")
    inp = {k: v.cuda() for k, v in si.decode_inputs(shape, 0, seed=2).items()}
    keep = [0, 1, 3]
    pool_a, cpool_a = pools["ssm_pool"].clone(), pools["conv_pool"].clone()
    pool_b, cpool_b = pools["ssm_pool"].clone(), pools["conv_pool"].clone()
    old = ssd.ssd_set_debug_checks(ssd.SSD_CHECK_DISTINCT_SLOTS)
    try:
        y = _decode_call(shape, prm, inp["xbc"], inp["dt_raw"], inp["z"], [2, 5, 2, 7],
                         pool_a, cpool_a)
        assert ssd.ssd_read_device_error() == ssd.SSD_ERR_DUPLICATE_SLOT
    finally:
        ssd.ssd_set_debug_checks(old)
    y_ref = _decode_call(shape, prm, inp["xbc"][keep].contiguous(), inp["dt_raw"][keep].contiguous(),
                         inp["z"][keep].contiguous(), [2, 5, 7], pool_b, cpool_b)
    assert ssd.ssd_read_device_error() == ssd.SSD_OK
    assert torch.equal(pool_a, pool_b) and torch.equal(cpool_a, cpool_b)
    assert torch.equal(y[keep], y_ref)
    assert torch.isnan(y[2].float()).all()


def test_duplicate_varlen_slot_reported_and_skipped_with_debug_checks():
    """Packed sequences at slots [3, 1, 3]: the third writes nothing (pools, y)
    and sets SSD_ERR_DUPLICATE_SLOT; the first two are bit for bit the call
    without it."""
    H, G, P, N, W = 8, 2, 64, 128, 4
    lens = [130, 40, 60]
    T = sum(lens)
    shape = si.Shape(batch=1, seqlen=T, nheads=H, headdim=P, dstate=N, ngroups=G)
    prm = {k: v.cuda() for k, v in si.params(shape, seed=4).items()}
    inp = si.prefill_inputs(shape, seed=4, device="cuda")
    rows = {k: inp[k][0].contiguous() for k in ("xbc", "dt_raw", "z")}
    g = torch.Generator(device="cuda").manual_seed(5)
    spool0 = torch.randn((5, H, P, N), generator=g, device="cuda") * 0.1
    cpool0 = torch.randn((5, W - 1, shape.cdim), generator=g, device="cuda").to(torch.bfloat16)
    flags = ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z

    def call(nseq, slots, spool, cpool):
        t = sum(lens[:nseq])
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens[:nseq])]), dtype=torch.int32,
                          device="cuda")
        y = torch.full((T, H, P), float("nan"), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(T * 2 * G * N * 2, dtype=torch.uint8, device="cuda")
        ssd.ssd_chunk_scan_varlen(
            ssd.dims(nseq, t, H, P, N, G, W), ssd.SSD_BF16, flags, cu,
            torch.tensor(slots, dtype=torch.int32, device="cuda"), None, 5, rows["xbc"][:t],
            prm["conv_w"], prm["conv_b"], cpool, rows["dt_raw"][:t], prm["dt_bias"], prm["A"],
            prm["D"], rows["z"][:t], spool, y[:t], ws)
        return y

    sa, ca = spool0.clone(), cpool0.clone()
    old = ssd.ssd_set_debug_checks(ssd.SSD_CHECK_DISTINCT_SLOTS)
    try:
        ya = call(3, [3, 1, 3], sa, ca)
        assert ssd.ssd_read_device_error() == ssd.SSD_ERR_DUPLICATE_SLOT
    finally:
        ssd.ssd_set_debug_checks(old)
    sb, cb = spool0.clone(), cpool0.clone()
    yb = call(2, [3, 1], sb, cb)
    assert ssd.ssd_read_device_error() == ssd.SSD_OK
    t2 = lens[0] + lens[1]
    assert torch.equal(sa, sb) and torch.equal(ca, cb)
    assert torch.equal(ya[:t2], yb[:t2])
    assert torch.isnan(ya[t2:].float()).all()
