"""GPU parity: the CUDA library (through the C-ABI) against the fp64 oracle.

Every test here runs the library's kernels on cuda:0 and compares with the
oracle on the same seeded inputs (tests/helpers.py states the tolerance).
"""
import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
from tests.helpers import (TOL, assert_close, check_prefill_every_element, f64, gpu_prefill,
                           make_problem, oracle_prefill, oracle_sequence)

pytestmark = pytest.mark.gpu

ssd = pytest.importorskip("ssd_scan_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ssd.load_library()
    yield
    assert ssd.ssd_read_device_error() == ssd.SSD_OK


def _check_prefill(shape, cpu, y, h, cs, act, conv=True, dt_softplus=True, heads=None,
                   batches=None):
    yo, ho, co, cols = oracle_prefill(shape, cpu, conv=conv, dt_softplus=dt_softplus,
                                      heads=heads, batches=batches)
    hh = list(range(shape.nheads)) if heads is None else list(heads)
    bb = list(range(shape.batch)) if batches is None else list(batches)
    tol = TOL[act]
    P, N = shape.headdim, shape.dstate
    e1 = assert_close(y[bb][:, :, hh], yo, tol, count=len(bb) * shape.seqlen * len(hh) * P,
                      what="y")
    e2 = assert_close(h[bb][:, hh], ho, tol, count=len(bb) * len(hh) * P * N, what="ssm_state")
    if conv and cs is not None:
        gcs = f64(cs)[bb][:, :, cols]
        assert np.array_equal(gcs, co), "conv state must be the raw rows, bit for bit"
    return e1, e2


# ---------------------------------------------------------------------------
# tiny fp32 problem: 11 rows in one call, as 7 + 4, and one row per call

@pytest.mark.parametrize("splits", [[11], [7, 4], [1] * 11, [3, 5, 3]])
@pytest.mark.parametrize("init", [False, True])
def test_tiny_fp32(splits, init):
    shape = si.TINY
    cpu, dev = make_problem(shape, act=torch.float32, initial_state=init, with_z=True)
    y, h, cs = gpu_prefill(shape, dev, splits)
    _check_prefill(shape, cpu, y, h, cs, torch.float32)


def test_tiny_fp32_no_conv_no_z_no_softplus():
    shape = si.TINY
    cpu, dev = make_problem(shape, act=torch.float32, with_z=False)
    dt = cpu["dt_raw"].abs() * 0.1  # dt taken as given: positive, moderate
    cpu["dt_raw"] = dt
    dev["dt_raw"] = dt.cuda()
    y, h, _ = gpu_prefill(shape, dev, [7, 4], conv=False, dt_softplus=False)
    _check_prefill(shape, cpu, y, h, None, torch.float32, conv=False, dt_softplus=False)


def test_dt_zero_leaves_state_bit_unchanged():
    shape = si.TINY
    cpu, dev = make_problem(shape, act=torch.float32)
    dev["dt_raw"] = torch.zeros_like(dev["dt_raw"])
    y, h, _ = gpu_prefill(shape, dev, [7, 4], conv=False, dt_softplus=False)
    assert torch.equal(h, dev["ssm_state"])


# ---------------------------------------------------------------------------
# conv alone

@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("S", [1, 2, 5, 200])
@pytest.mark.parametrize("inplace", [False, True])
def test_conv1d_rows(act, S, inplace):
    shape = si.TINY.with_(batch=3, seqlen=S)
    cpu, dev = make_problem(shape, act=act)
    C, W = shape.cdim, shape.conv_width
    d = ssd.dims(3, S, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, W)
    out = torch.empty_like(dev["xbc"])
    st_in = dev["conv_state"].clone()
    st_out = st_in if inplace else torch.empty_like(st_in)
    ssd.ssd_conv1d_rows(d, ssd.act_of(out), dev["xbc"], dev["conv_w"], dev["conv_b"], st_in,
                        out, st_out)
    ref, ref_st = oracle.conv1d(f64(cpu["xbc"]), f64(cpu["conv_w"]), f64(cpu["conv_b"]),
                                f64(cpu["conv_state"]))
    assert_close(out, ref, TOL[act], count=3 * S * C, what="conv out")
    assert np.array_equal(f64(st_out), ref_st)


# ---------------------------------------------------------------------------
# bf16 prefill at small sizes that span several 128-row chunks + ragged tail

@pytest.mark.parametrize("splits", [[300], [128, 172], [37, 91, 172], [1, 299]])
def test_prefill_bf16_multichunk(splits):
    shape = si.Shape(batch=2, seqlen=300, nheads=8, headdim=64, dstate=128, ngroups=2)
    cpu, dev = make_problem(shape, act=torch.bfloat16)
    y, h, cs = gpu_prefill(shape, dev, splits)
    _check_prefill(shape, cpu, y, h, cs, torch.bfloat16)


def test_prefill_bf16_fresh_request_no_z():
    shape = si.Shape(batch=1, seqlen=137, nheads=4, headdim=64, dstate=128, ngroups=1)
    cpu, dev = make_problem(shape, act=torch.bfloat16, initial_state=False, with_z=False)
    y, h, cs = gpu_prefill(shape, dev)
    _check_prefill(shape, cpu, y, h, cs, torch.bfloat16)


def test_prefill_empty_rows_copies_state():
    shape = si.Shape(batch=2, seqlen=0, nheads=4, headdim=64, dstate=128, ngroups=1)
    cpu, dev = make_problem(shape, act=torch.bfloat16)
    y, h, cs = gpu_prefill(shape, dev)
    assert y.numel() == 0
    assert torch.equal(h, dev["ssm_state"])
    assert torch.equal(cs, dev["conv_state"])


def test_decay_stress_small():
    shape = si.Shape(batch=2, seqlen=260, nheads=4, headdim=64, dstate=128, ngroups=1)
    cpu, dev = make_problem(shape, act=torch.bfloat16, stress=True)
    splits = si.random_splits(260, seed=3)
    y, h, cs = gpu_prefill(shape, dev, splits)
    assert torch.isfinite(y.float()).all() and torch.isfinite(h).all()
    _check_prefill(shape, cpu, y, h, cs, torch.bfloat16)


# ---------------------------------------------------------------------------
# Nemotron-H-8B-shaped prefill at full size: B=1, S=2048, H=128; every
# element of y and of the final states against the oracle

def test_prefill_full_size_every_element():
    shape = si.PREFILL
    cpu, dev = make_problem(shape, act=torch.bfloat16)
    y, h, cs = gpu_prefill(shape, dev)
    check_prefill_every_element(shape, cpu, y, h, cs, torch.bfloat16)


def test_prefill_137_rows_every_element():
    shape = si.PREFILL.with_(seqlen=137)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=5, initial_state=False)
    y, h, cs = gpu_prefill(shape, dev)
    check_prefill_every_element(shape, cpu, y, h, cs, torch.bfloat16)


@pytest.mark.parametrize("B,S", [(3, 100), (2, 5), (4, 128), (1, 77)])
def test_short_calls_several_units_per_cta_every_element(B, S):
    """Calls of at most 128 rows run on the kernel whose CTAs walk several
    (sequence, head) units each: 128 heads x B sequences over the SMs, so most
    CTAs take two or more units (one at B = 1).  Every element of y and of the
    final states against the oracle, the conv state bit for bit."""
    shape = si.PREFILL.with_(batch=B, seqlen=S)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=17 + S)
    before = ssd.ssd_launch_counts()
    y, h, cs = gpu_prefill(shape, dev)
    after = ssd.ssd_launch_counts()
    assert after["scan_tc"] - before["scan_tc"] == 1 and after["scan_simt"] == before["scan_simt"]
    check_prefill_every_element(shape, cpu, y, h, cs, torch.bfloat16)


@pytest.mark.parametrize("splits", [[129, 130, 258], [1, 128, 2, 386]])
def test_calls_whose_last_chunk_is_short_chain_their_conv_state(splits):
    """Calls whose last chunk holds 1 or 2 rows: the new conv state (the last
    W-1 raw rows) then reaches back into the chunk before.  Chained calls over
    517 rows, every element of y and of the final states against one oracle
    pass over all rows (a wrong conv state would also corrupt the next call's
    first rows); the final conv state bit for bit."""
    shape = si.Shape(batch=2, seqlen=sum(splits), nheads=16, headdim=64, dstate=128, ngroups=2)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=13)
    y, h, cs = gpu_prefill(shape, dev, splits)
    check_prefill_every_element(shape, cpu, y, h, cs, torch.bfloat16)


@pytest.mark.parametrize("S", [1, 2, 3, 77, 128, 129, 300])
def test_states_updated_in_place_equal_separate_outputs(S):
    """The final states may be written over the initial ones (conv_state_out
    = conv_state_in, ssm_state_out = ssm_state_in): y and both states equal,
    bit for bit, those of the same call with separate outputs -- on the
    multi-unit kernel (S <= 128) and on the chunk kernel, and for S < W-1,
    where the new conv state keeps rows of the old one."""
    shape = si.Shape(batch=3, seqlen=S, nheads=16, headdim=64, dstate=128, ngroups=2)
    _, dev = make_problem(shape, act=torch.bfloat16, seed=40 + S)
    kw = dict(nheads=16, headdim=64, dstate=128, ngroups=2, conv_w=dev["conv_w"],
              conv_b=dev["conv_b"], dt_bias=dev["dt_bias"], D=dev["D"], z=dev["z"])
    y1, h1, c1 = ssd.chunk_scan(dev["xbc"], dev["dt_raw"], dev["A"], conv_state=dev["conv_state"],
                                ssm_state=dev["ssm_state"], **kw)
    hs, cs = dev["ssm_state"].clone(), dev["conv_state"].clone()
    y2 = torch.empty_like(y1)
    ssd.chunk_scan(dev["xbc"], dev["dt_raw"], dev["A"], conv_state=cs, ssm_state=hs,
                   out=(y2, hs, cs), **kw)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2), "y"
    assert torch.equal(h1, hs), "ssm state written in place"
    assert torch.equal(c1, cs), "conv state written in place"


# ---------------------------------------------------------------------------
# the other workloads at full size, in the calls the benchmark makes.  Inputs
# are drawn on the GPU; the checked sequences are copied to the host and the
# oracle runs one (sequence, group of heads) at a time.

def _device_problem(shape, seed, stress=False):
    prm = si.params(shape, seed=seed, stress=stress)
    inp = si.prefill_inputs(shape, seed=seed, device="cuda", stress=stress)
    dev = {**{k: v.cuda() for k, v in prm.items()}, **inp}
    return prm, inp, dev


def _host_subset(prm, inp, batches):
    sub = {k: (v[batches].cpu() if v is not None else None) for k, v in inp.items()}
    return {**prm, **sub}


def test_long_prefill_full_size_chained_every_element():
    """8 sequences x 8192 rows, then a second 8192-row call fed with the first
    call's final states, on all 128 heads; every element of two sequences
    (all heads, all 16384 rows, both final states) against the oracle, and
    every output finite."""
    shape = si.LONG.with_(seqlen=2 * si.LONG.seqlen)
    prm, inp, dev = _device_problem(shape, seed=11)
    y, h, cs = gpu_prefill(shape, dev, [si.LONG.seqlen, si.LONG.seqlen])
    assert torch.isfinite(y.float()).all() and torch.isfinite(h).all()
    bb = [0, 7]
    cpu = _host_subset(prm, inp, bb)
    del inp, dev
    check_prefill_every_element(shape.with_(batch=len(bb)), cpu, y, h, cs, torch.bfloat16,
                                gpu_batch_of=bb)


def test_decay_stress_full_size_every_element():
    """4 sequences x 4096 rows with decays up to ~1e4 per row, fed as calls of
    U{1..128} rows, one split shared by the batch: every element against the
    oracle."""
    shape = si.STRESS
    prm, inp, dev = _device_problem(shape, seed=13, stress=True)
    y, h, cs = gpu_prefill(shape, dev, si.random_splits(shape.seqlen, seed=13))
    assert torch.isfinite(y.float()).all() and torch.isfinite(h).all()
    cpu = _host_subset(prm, inp, list(range(shape.batch)))
    check_prefill_every_element(shape, cpu, y, h, cs, torch.bfloat16)


def test_decay_stress_independent_splits_per_sequence():
    """The same stress sequences, each on its own (batch 1): once with its own
    seeded split of U{1..128}-row calls and once as one 4096-row call.  Both
    against the oracle, every element; and the shared-split batched run too.
    (One long call is where every chunk's total decay is ~1e6: gamma_Q must be
    the last row's own cumulative-sum value, converted to log2 units without
    losing its low part, or the final state is off by several percent.)"""
    shape = si.STRESS
    prm, inp, dev = _device_problem(shape, seed=13, stress=True)
    yb, hb, _ = gpu_prefill(shape, dev, si.random_splits(shape.seqlen, seed=13))
    one = shape.with_(batch=1)
    tol = TOL[torch.bfloat16]
    n_y, n_h = shape.seqlen * shape.nheads * shape.headdim, shape.nheads * 64 * 128
    for b in range(shape.batch):
        dev1 = {k: (v[b:b + 1].contiguous() if (k in inp and v is not None) else v)
                for k, v in dev.items()}
        cpu = _host_subset(prm, inp, [b])
        yo, ho = oracle_sequence(one, cpu, 0)
        ys, hs, _ = gpu_prefill(one, dev1, si.random_splits(shape.seqlen, seed=100 + b))
        y1, h1, _ = gpu_prefill(one, dev1)  # the whole sequence in one call
        for what, yy, hh in (("split", ys[0], hs[0]), ("one call", y1[0], h1[0]),
                             ("batched", yb[b], hb[b])):
            assert_close(yy, yo, tol, count=n_y, what=f"seq {b} y ({what})")
            assert_close(hh, ho, tol, count=n_h, what=f"seq {b} state ({what})")


def test_prefill_eight_heads_per_group():
    """The 30B-A3B mixer shape: 64 heads of 64 in 8 groups of state size 128
    (8 heads per group), bf16, over two calls."""
    shape = si.Shape(batch=2, seqlen=300, nheads=64, headdim=64, dstate=128, ngroups=8)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=17)
    y, h, cs = gpu_prefill(shape, dev, [200, 100])
    _check_prefill(shape, cpu, y, h, cs, torch.bfloat16, heads=[0, 7, 8, 33, 63])


# ---------------------------------------------------------------------------
# which kernels ran (launch counters), and the paths around the tensor cores

def _counts():
    return ssd.ssd_launch_counts()


def test_bf16_runs_on_tensor_cores():
    shape = si.Shape(batch=1, seqlen=256, nheads=8, headdim=64, dstate=128, ngroups=2)
    cpu, dev = make_problem(shape, act=torch.bfloat16)
    c0 = _counts()
    y, h, cs = gpu_prefill(shape, dev)
    torch.cuda.synchronize()
    c1 = _counts()
    assert c1["scan_tc"] - c0["scan_tc"] == 1
    assert c1["bc_conv"] - c0["bc_conv"] == 1
    assert c1["scan_simt"] == c0["scan_simt"]
    _check_prefill(shape, cpu, y, h, cs, torch.bfloat16)


def test_bf16_calls_of_a_few_rows_run_on_tensor_cores():
    """Calls of 1 to 5 rows run on the tensor cores too (their units walk the
    chunk pipeline several per CTA), chained into one sequence."""
    shape = si.Shape(batch=2, seqlen=12, nheads=8, headdim=64, dstate=128, ngroups=2)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=4)
    c0 = _counts()
    y, h, cs = gpu_prefill(shape, dev, [1, 2, 4, 5])
    torch.cuda.synchronize()
    c1 = _counts()
    assert c1["scan_tc"] - c0["scan_tc"] == 4 and c1["scan_simt"] == c0["scan_simt"]
    _check_prefill(shape, cpu, y, h, cs, torch.bfloat16)


def test_bf16_tensor_cores_without_conv():
    shape = si.Shape(batch=2, seqlen=200, nheads=4, headdim=64, dstate=128, ngroups=2)
    cpu, dev = make_problem(shape, act=torch.bfloat16)
    c0 = _counts()
    y, h, _ = gpu_prefill(shape, dev, [77, 123], conv=False)
    torch.cuda.synchronize()
    c1 = _counts()
    assert c1["scan_tc"] - c0["scan_tc"] == 2 and c1["bc_conv"] == c0["bc_conv"]
    _check_prefill(shape, cpu, y, h, None, torch.bfloat16, conv=False)


def test_bf16_other_head_dims_run_row_exact_kernel():
    shape = si.Shape(batch=1, seqlen=150, nheads=4, headdim=32, dstate=64, ngroups=1)
    cpu, dev = make_problem(shape, act=torch.bfloat16)
    c0 = _counts()
    y, h, cs = gpu_prefill(shape, dev, [100, 50])
    torch.cuda.synchronize()
    c1 = _counts()
    assert c1["scan_simt"] - c0["scan_simt"] == 2 and c1["scan_tc"] == c0["scan_tc"]
    _check_prefill(shape, cpu, y, h, cs, torch.bfloat16)


@pytest.mark.parametrize("W", [2, 3])
@pytest.mark.parametrize("splits", [[130, 130], [100, 1, 59, 100]])
def test_bf16_short_conv_widths(W, splits):
    """Conv widths below 4 on the tensor-core paths: calls of more than one
    chunk (the chunk kernel) and of at most 128 rows (the multi-unit kernel,
    whose taps are front-padded to 4), chained."""
    shape = si.Shape(batch=2, seqlen=260, nheads=4, headdim=64, dstate=128, ngroups=1,
                     conv_width=W)
    cpu, dev = make_problem(shape, act=torch.bfloat16)
    y, h, cs = gpu_prefill(shape, dev, splits)
    _check_prefill(shape, cpu, y, h, cs, torch.bfloat16)


def test_mixed_magnitude_decay_in_one_chunk():
    """One row with a decay of ~e^-1000 followed by rows of small decay in the
    same chunk: gamma differences of small rows after the big one must keep
    their precision (double-float cumulative sum)."""
    shape = si.Shape(batch=1, seqlen=256, nheads=4, headdim=64, dstate=128, ngroups=1)
    cpu, dev = make_problem(shape, act=torch.bfloat16)
    dt_raw = cpu["dt_raw"].clone()
    dt_raw[0, 40, :] = 300.0     # dt ~ 300 at row 40 -> dt*A ~ -300..-4800
    dt_raw[0, 170, :] = 120.0    # and one in the second chunk
    cpu["dt_raw"] = dt_raw
    dev["dt_raw"] = dt_raw.cuda()
    y, h, cs = gpu_prefill(shape, dev)
    assert torch.isfinite(y.float()).all() and torch.isfinite(h).all()
    _check_prefill(shape, cpu, y, h, cs, torch.bfloat16)


@pytest.mark.parametrize("scale", [0.25, 1.0, 4.0, 16.0])
def test_decay_range_across_factored_threshold(scale):
    """Chunks whose total decay falls on either side of the range where the
    mask factors into exp(gamma_t) exp(-gamma_s) give the same answer."""
    shape = si.Shape(batch=1, seqlen=384, nheads=8, headdim=64, dstate=128, ngroups=2)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=7)
    cpu["A"] = cpu["A"] * scale
    dev["A"] = cpu["A"].cuda()
    y, h, cs = gpu_prefill(shape, dev)
    _check_prefill(shape, cpu, y, h, cs, torch.bfloat16)


@pytest.mark.parametrize("row", [0, 31, 32, 63, 95, 127])
def test_exact_chunk_decay_spike_at_block_edges(row):
    """A spike of decay (~e^-300 per head) at a row on either side of a 32-row
    block edge of the mask: the exact form splits the decay of the blocks below
    the diagonal at their last row, so a spike there must land on the right
    side of the split."""
    shape = si.Shape(batch=1, seqlen=200, nheads=4, headdim=64, dstate=128, ngroups=1)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=11)
    dt_raw = cpu["dt_raw"].clone()
    dt_raw[0, row, :] = 60.0
    dt_raw[0, 128 + row // 2, :] = 40.0  # and one in the second, ragged chunk
    cpu["dt_raw"] = dt_raw
    dev["dt_raw"] = dt_raw.cuda()
    y, h, cs = gpu_prefill(shape, dev, [70, 130])
    assert torch.isfinite(y.float()).all() and torch.isfinite(h).all()
    _check_prefill(shape, cpu, y, h, cs, torch.bfloat16)


def test_exact_chunk_rising_and_falling_gamma():
    """dt taken as given (no softplus) with negative entries: gamma rises and
    falls inside a chunk.  The chunk form then differs from the row recurrence
    (each exponent is clamped at 0), so the reference is the oracle's chunk
    form over the same 128-row chunks; no column block may split its decay at
    a middle row here (the clamps do not factor)."""
    shape = si.Shape(batch=1, seqlen=256, nheads=4, headdim=64, dstate=128, ngroups=1)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=13)
    g = torch.Generator().manual_seed(5)
    dt_raw = torch.rand(cpu["dt_raw"].shape, generator=g) * 0.2 - 0.05  # [-0.05, 0.15)
    cpu["dt_raw"] = dt_raw
    dev["dt_raw"] = dt_raw.cuda()
    y, h, cs = gpu_prefill(shape, dev, dt_softplus=False)
    assert torch.isfinite(y.float()).all() and torch.isfinite(h).all()
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    xbc, _ = oracle.conv1d(f64(cpu["xbc"]), f64(cpu["conv_w"]), f64(cpu["conv_b"]),
                           f64(cpu.get("conv_state")), apply_silu=True)
    yo, ho = oracle.ssd_chunked(xbc, f64(dt_raw), f64(cpu["A"]), [128, 128], H=H, P=P, N=N, G=G,
                                dt_bias=f64(cpu["dt_bias"]), D=f64(cpu["D"]), z=f64(cpu.get("z")),
                                h0=f64(cpu.get("ssm_state")), dt_softplus=False)
    assert_close(y, yo, TOL[torch.bfloat16], count=y.numel(), what="y")
    assert_close(h, ho, TOL[torch.bfloat16], count=h.numel(), what="ssm_state")
