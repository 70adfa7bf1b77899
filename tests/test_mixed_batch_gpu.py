"""A mixed prefill + decode batch on shared state pools (vllm.cpp #1362
summary: the prefill half of a batch runs the chunk scan over packed rows with
states at the state index, the decode half the single-step kernel at its slots;
which half a request belongs to is the metadata's decode count, never its token
count, so a one-token prefill of a fresh request still takes the chunk scan).

Two steps on one SSM pool and one conv pool: each step sends packed prefill
sequences (a 1-row fresh request among them) through ssd_chunk_scan_varlen and
decode rows at other slots through ssd_decode_step.  Step 2 turns step 1's
prefills into decodes and continues a decoded slot with a 5-token prefill.
Every y and every touched slot is compared with the oracle's
mixer_prefill_varlen followed by mixer_decode; untouched slots must be
bit-identical."""
import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
from tests.helpers import TOL, assert_close, f64

pytestmark = pytest.mark.gpu

ssd = pytest.importorskip("ssd_scan_gb300")

SHAPE = si.Shape(batch=1, seqlen=1, nheads=16, headdim=64, dstate=128, ngroups=2)
NSLOTS = 12
# (prefill lengths, prefill slots, has_initial_state, decode slots) per step
STEPS = [
    ([1, 200, 130], [4, 9, 0], [0, 1, 0], [2, 7, 11, 5, 3]),
    ([3, 5], [1, 2], [0, 1], [4, 9, 0, 7]),
]
UNTOUCHED = [6, 8, 10]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ssd.load_library()
    yield
    assert ssd.ssd_read_device_error() == ssd.SSD_OK


def _rows(n, g):
    H, P, C = SHAPE.nheads, SHAPE.headdim, SHAPE.cdim
    return {"xbc": torch.randn((n, C), generator=g).to(torch.bfloat16),
            "dt_raw": torch.randn((n, H), generator=g),
            "z": torch.randn((n, H * P), generator=g).to(torch.bfloat16)}


def test_mixed_prefill_and_decode_batch_on_shared_pools():
    H, P, N, G, W = SHAPE.nheads, SHAPE.headdim, SHAPE.dstate, SHAPE.ngroups, SHAPE.conv_width
    prm = si.params(SHAPE, seed=3)
    g = torch.Generator().manual_seed(41)
    spool0 = torch.randn((NSLOTS, H, P, N), generator=g) * 0.1
    cpool0 = torch.randn((NSLOTS, W - 1, SHAPE.cdim), generator=g).to(torch.bfloat16)
    dev = torch.device("cuda")
    dprm = {k: v.to(dev) for k, v in prm.items()}
    spool, cpool = spool0.to(dev), cpool0.to(dev)
    o_spool, o_cpool = f64(spool0), f64(cpool0)
    flags = ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z
    kw = dict(H=H, P=P, N=N, G=G, conv_b=f64(prm["conv_b"]), dt_bias=f64(prm["dt_bias"]),
              D=f64(prm["D"]))
    for lens, pslots, init, dslots in STEPS:
        T, R = sum(lens), len(dslots)
        pre, dec = _rows(T, g), _rows(R, g)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        c0 = ssd.ssd_launch_counts()
        # prefill half: packed rows through the chunk scan, states at the slots
        y_p = torch.full((T, H, P), float("nan"), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(T * 2 * G * N * 2, dtype=torch.uint8, device=dev)
        ssd.ssd_chunk_scan_varlen(
            ssd.dims(len(lens), T, H, P, N, G, W), ssd.SSD_BF16, flags,
            torch.from_numpy(cu).to(dev), torch.tensor(pslots, dtype=torch.int32, device=dev),
            torch.tensor(init, dtype=torch.int32, device=dev), NSLOTS, pre["xbc"].to(dev),
            dprm["conv_w"], dprm["conv_b"], cpool, pre["dt_raw"].to(dev), dprm["dt_bias"],
            dprm["A"], dprm["D"], pre["z"].to(dev), spool, y_p, ws)
        # decode half: one token per row at its slot, in place, same pools
        y_d = torch.full((R, H, P), float("nan"), dtype=torch.bfloat16, device=dev)
        ssd.ssd_decode_step(
            ssd.dims(R, 1, H, P, N, G, W), ssd.SSD_BF16, flags, dec["xbc"].to(dev),
            dprm["conv_w"], dprm["conv_b"], cpool, dec["dt_raw"].to(dev), dprm["dt_bias"],
            dprm["A"], dprm["D"], dec["z"].to(dev),
            torch.tensor(dslots, dtype=torch.int32, device=dev), NSLOTS, spool, y_d)
        torch.cuda.synchronize()
        c1 = ssd.ssd_launch_counts()
        # the 1-row fresh request went through the chunk scan, not the row kernel
        assert c1["scan_tc"] - c0["scan_tc"] == 1 and c1["scan_simt"] == c0["scan_simt"]
        assert c1["decode_step"] - c0["decode_step"] == 1
        # oracle: the prefill half, then the decode half on the pools it left
        yo_p, o_spool, o_cpool = oracle.mixer_prefill_varlen(
            f64(pre["xbc"]), f64(prm["conv_w"]), f64(pre["dt_raw"]), f64(prm["A"]), cu, pslots,
            o_spool, o_cpool, has_initial_state=init, z=f64(pre["z"]), **kw)
        yo_d, o_spool, o_cpool = oracle.mixer_decode(
            f64(dec["xbc"]), f64(prm["conv_w"]), f64(dec["dt_raw"]), f64(prm["A"]), dslots,
            o_spool, conv_pool=o_cpool, z=f64(dec["z"]), **kw)
        tol = TOL[torch.bfloat16]
        assert_close(y_p, yo_p, tol, count=T * H * P, what="prefill y")
        assert_close(y_d, yo_d, tol, count=R * H * P, what="decode y")
        for s in pslots + dslots:
            assert_close(spool[s], o_spool[s], tol, count=H * P * N, what=f"slot {s}")
            assert np.array_equal(f64(cpool[s]), o_cpool[s]), f"conv state of slot {s}"
    for s in UNTOUCHED:
        assert torch.equal(spool[s].cpu(), spool0[s]) and torch.equal(cpool[s].cpu(), cpool0[s])
