"""GPU parity of the scan over packed sequences with slot-indexed states
(ssd_chunk_scan_varlen; vllm.cpp #1362 summary, TensorSharp "nemotron.md"
section 11) through the C-ABI, against the fp64 oracle on the same stored
inputs; tolerance as in tests/helpers.py, raw conv-state rows bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
from tests.helpers import TOL, MaxRel, assert_close, f64

pytestmark = pytest.mark.gpu

ssd = pytest.importorskip("ssd_scan_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ssd.load_library()
    yield
    assert ssd.ssd_read_device_error() == ssd.SSD_OK


def _problem(lens, nslots, H=8, G=2, seed=0):
    shape = si.Shape(batch=1, seqlen=max(1, sum(lens)), nheads=H, headdim=64, dstate=128,
                     ngroups=G)
    prm = si.params(shape, seed=seed)
    inp = si.prefill_inputs(shape, seed=seed, with_z=True)
    T = sum(lens)
    rows = {k: inp[k][0, :T].contiguous() for k in ("xbc", "dt_raw", "z")}
    g = torch.Generator().manual_seed(seed + 1)
    spool = torch.randn((nslots, H, 64, 128), generator=g) * 0.1
    cpool = torch.randn((nslots, shape.conv_width - 1, shape.cdim), generator=g).to(torch.bfloat16)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    return shape, prm, rows, spool, cpool, cu


def _run_gpu(shape, prm, rows, spool, cpool, cu, slots, init, num_slots=None):
    dev = torch.device("cuda")
    H, P, N, G, W = shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.conv_width
    nseq, T = len(slots), rows["xbc"].shape[0]
    d = ssd.dims(nseq, T, H, P, N, G, W)
    sp, cp = spool.to(dev), cpool.to(dev)
    y = torch.full((T, H, P), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(1, T * 2 * G * N * 2), dtype=torch.uint8, device=dev)
    ssd.ssd_chunk_scan_varlen(
        d, ssd.SSD_BF16, ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z, cu.to(dev),
        torch.tensor(slots, dtype=torch.int32, device=dev),
        None if init is None else torch.tensor(init, dtype=torch.int32, device=dev),
        num_slots or spool.shape[0], rows["xbc"].to(dev), prm["conv_w"].to(dev),
        prm["conv_b"].to(dev), cp, rows["dt_raw"].to(dev), prm["dt_bias"].to(dev),
        prm["A"].to(dev), prm["D"].to(dev), rows["z"].to(dev), sp, y, ws)
    return y, sp, cp


def _run_oracle(shape, prm, rows, spool, cpool, cu, slots, init, heads=None):
    H = shape.nheads
    return oracle.mixer_prefill_varlen(
        f64(rows["xbc"]), f64(prm["conv_w"]), f64(rows["dt_raw"]), f64(prm["A"]), cu.numpy(),
        slots, f64(spool), f64(cpool), H=H, P=shape.headdim, N=shape.dstate, G=shape.ngroups,
        has_initial_state=init, conv_b=f64(prm["conv_b"]), dt_bias=f64(prm["dt_bias"]),
        D=f64(prm["D"]), z=f64(rows["z"]))


def test_varlen_mixed_lengths_and_slots_match_oracle():
    """Empty, 1-row, chunk-edge (127/128/129) and multi-chunk sequences at
    permuted slots, fresh and continuing; slots no sequence names stay
    bit-identical."""
    lens = [0, 1, 127, 128, 129, 300, 5]
    slots = [9, 3, 0, 7, 5, 1, 8]
    init = [1, 1, 0, 1, 1, 0, 1]
    shape, prm, rows, spool, cpool, cu = _problem(lens, nslots=10)
    y, sp, cp = _run_gpu(shape, prm, rows, spool, cpool, cu, slots, init)
    yo, spo, cpo = _run_oracle(shape, prm, rows, spool, cpool, cu, slots, init)
    T, H, P = yo.shape
    assert_close(y, yo, TOL[torch.bfloat16], count=T * H * P, what="y")
    for s in slots:
        assert_close(sp[s], spo[s], TOL[torch.bfloat16], count=H * P * 128, what=f"slot {s}")
        assert np.array_equal(f64(cp[s]), cpo[s]), f"conv state of slot {s}"
    for s in (2, 4, 6):
        assert torch.equal(sp[s].cpu(), spool[s]) and torch.equal(cp[s].cpu(), cpool[s])


def test_varlen_equal_lengths_reproduce_the_batched_call():
    """Equal lengths at slots 0..B-1 continuing their states: bit for bit the
    batched ssd_chunk_scan (the same kernel, only its row and state offsets
    differ)."""
    B, S = 3, 200
    shape, prm, rows, spool, cpool, cu = _problem([S] * B, nslots=B, seed=4)
    y, sp, cp = _run_gpu(shape, prm, rows, spool, cpool, cu, [0, 1, 2], None)
    d = ssd.dims(B, S, shape.nheads, 64, 128, shape.ngroups, shape.conv_width)
    dev = torch.device("cuda")
    yb, hb, cb = ssd.chunk_scan(
        rows["xbc"].reshape(B, S, -1).to(dev), rows["dt_raw"].reshape(B, S, -1).to(dev),
        prm["A"].to(dev), nheads=shape.nheads, headdim=64, dstate=128, ngroups=shape.ngroups,
        conv_w=prm["conv_w"].to(dev), conv_b=prm["conv_b"].to(dev), conv_state=cpool.to(dev),
        dt_bias=prm["dt_bias"].to(dev), D=prm["D"].to(dev),
        z=rows["z"].reshape(B, S, -1).to(dev), ssm_state=spool.to(dev))
    assert torch.equal(y.reshape(B, S, shape.nheads, 64), yb)
    assert torch.equal(sp, hb) and torch.equal(cp, cb)


def test_varlen_full_width_every_element():
    """The Nemotron-H-8B heads (128 heads, 8 groups): a long, a medium, a short
    and a one-row sequence at permuted slots, fresh and continuing; every y
    element and every touched slot against the oracle, one group of 16 heads
    (with its own B|C columns) at a time."""
    lens = [2048, 600, 77, 1]
    slots = [2, 0, 3, 1]
    init = [1, 0, 1, 1]
    shape, prm, rows, spool, cpool, cu = _problem(lens, nslots=4, H=128, G=8, seed=6)
    y, sp, cp = _run_gpu(shape, prm, rows, spool, cpool, cu, slots, init)
    H, P, N, G = 128, 64, 128, 8
    hpg = H // G
    ey, eh = MaxRel("y"), MaxRel("slots")
    for g in range(G):
        heads = list(range(g * hpg, (g + 1) * hpg))
        cols = np.concatenate([np.arange(g * hpg * P, (g + 1) * hpg * P),
                               np.arange(H * P + g * N, H * P + (g + 1) * N),
                               np.arange(H * P + G * N + g * N, H * P + G * N + (g + 1) * N)])
        zc = np.arange(g * hpg * P, (g + 1) * hpg * P)
        sub_rows = {"xbc": rows["xbc"][:, cols], "dt_raw": rows["dt_raw"][:, heads],
                    "z": rows["z"][:, zc]}
        sub_prm = {"conv_w": prm["conv_w"][cols], "conv_b": prm["conv_b"][cols],
                   "dt_bias": prm["dt_bias"][heads], "A": prm["A"][heads], "D": prm["D"][heads]}
        sub_shape = si.Shape(batch=1, seqlen=sum(lens), nheads=hpg, headdim=P, dstate=N,
                             ngroups=1)
        yo, spo, cpo = _run_oracle(sub_shape, sub_prm, sub_rows, spool[:, heads],
                                   cpool[:, :, cols], cu, slots, init)
        ey.add(y[:, g * hpg:(g + 1) * hpg], yo)
        for s in slots:
            eh.add(sp[s, g * hpg:(g + 1) * hpg], spo[s])
            assert np.array_equal(f64(cp[s])[:, cols], cpo[s])
    ey.check(TOL[torch.bfloat16], sum(lens) * H * P)
    eh.check(TOL[torch.bfloat16], len(slots) * H * P * N)


def test_varlen_bad_slot_sets_error_and_writes_nothing_for_it():
    lens = [40, 70]
    shape, prm, rows, spool, cpool, cu = _problem(lens, nslots=4, seed=8)
    y, sp, cp = _run_gpu(shape, prm, rows, spool, cpool, cu, [1, 9], [1, 1])
    assert ssd.ssd_read_device_error() == ssd.SSD_ERR_BAD_SLOT
    assert torch.isnan(y[40:].float()).all(), "the bad sequence wrote rows"
    for s in (0, 2, 3):
        assert torch.equal(sp[s].cpu(), spool[s]) and torch.equal(cp[s].cpu(), cpool[s])
    yo, spo, cpo = _run_oracle(shape, prm, {k: v[:40] for k, v in rows.items()}, spool, cpool,
                               cu[:2], [1], [1])
    assert_close(y[:40], yo, TOL[torch.bfloat16], count=40 * shape.nheads * 64, what="y")


def test_varlen_no_rows_zeroes_fresh_slots_only():
    """Only empty sequences: a fresh one's states become zeros, a continuing
    one's stay as they were."""
    shape, prm, rows, spool, cpool, cu = _problem([0, 0], nslots=3, seed=10)
    y, sp, cp = _run_gpu(shape, prm, rows, spool, cpool, cu, [2, 0], [0, 1])
    assert torch.count_nonzero(sp[2]) == 0 and torch.count_nonzero(cp[2]) == 0
    assert torch.equal(sp[0].cpu(), spool[0]) and torch.equal(cp[0].cpu(), cpool[0])
    assert torch.equal(sp[1].cpu(), spool[1]) and torch.equal(cp[1].cpu(), cpool[1])
