"""GPU tests of ssd_decode_step: parity with the oracle and bit-exact slot
indexing (untouched slots unchanged, permutation invariance, in-place update
equal to a gathered contiguous copy), plus the bad-slot error word."""
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


def _setup(shape, num_slots, seed=0, act=torch.bfloat16, with_z=True):
    prm = {k: v.cuda() for k, v in si.params(shape, seed=seed).items()}
    pools = si.decode_pools(shape, num_slots, seed=seed, act_dtype=act, device="cuda")
    return prm, pools


def _step(shape, prm, pools, inp, conv=True, slots=None, pool=None, conv_pool=None,
          with_z=True):
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    R = inp["xbc"].shape[0]
    d = ssd.dims(R, 1, H, P, N, G, shape.conv_width)
    y = torch.empty((R, H, P), dtype=inp["xbc"].dtype, device="cuda")
    flags = ssd.SSD_DT_SOFTPLUS | (ssd.SSD_HAS_Z if with_z else 0)
    pool = pools["ssm_pool"] if pool is None else pool
    cpool = pools["conv_pool"] if conv_pool is None else conv_pool
    slots = pools["slot_ids"] if slots is None else slots
    ssd.ssd_decode_step(d, ssd.act_of(inp["xbc"]), flags, inp["xbc"],
                        prm["conv_w"] if conv else None, prm["conv_b"] if conv else None,
                        cpool if conv else None, inp["dt_raw"], prm["dt_bias"], prm["A"],
                        prm["D"], inp["z"] if with_z else None, slots, pool.shape[0], pool, y)
    return y


def _inputs(shape, step, seed=0, act=torch.bfloat16):
    return {k: (v.cuda() if v is not None else None)
            for k, v in si.decode_inputs(shape, step, seed=seed, act_dtype=act).items()}


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("conv", [True, False])
def test_decode_matches_oracle_over_steps(act, conv):
    shape = si.Shape(batch=12, seqlen=1, nheads=8, headdim=64, dstate=128, ngroups=2)
    prm, pools = _setup(shape, 40, act=act)
    pool0 = pools["ssm_pool"].clone()
    cpool0 = pools["conv_pool"].clone()
    steps = 5
    ys, ins = [], []
    for t in range(steps):
        inp = _inputs(shape, t, act=act)
        ins.append(inp)
        ys.append(_step(shape, prm, pools, inp, conv=conv))
    slots = pools["slot_ids"].cpu().numpy()
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    # the oracle: each row continues the sequence held in its slot
    xbc_seq = np.stack([f64(i["xbc"]) for i in ins], axis=1)      # [R, steps, C]
    dt_seq = np.stack([f64(i["dt_raw"]) for i in ins], axis=1)    # [R, steps, H]
    z_seq = np.stack([f64(i["z"]) for i in ins], axis=1)
    y_o, h_o, c_o = oracle.mixer_prefill(
        xbc_seq, f64(prm["conv_w"]) if conv else None, dt_seq, f64(prm["A"]), H=H, P=P, N=N,
        G=G, conv_b=f64(prm["conv_b"]) if conv else None,
        conv_state=f64(cpool0)[slots] if conv else None, dt_bias=f64(prm["dt_bias"]),
        D=f64(prm["D"]), z=z_seq, h0=f64(pool0)[slots])
    y_gpu = torch.stack(ys, dim=1)  # [R, steps, H, P]
    tol = TOL[act]
    assert_close(y_gpu, y_o, tol, count=12 * steps * H * P, what="y")
    assert_close(pools["ssm_pool"][pools["slot_ids"].long()], h_o, tol, what="pool")
    if conv:
        assert np.array_equal(f64(pools["conv_pool"])[slots], c_o)


def test_untouched_slots_and_permutation_bit_exact():
    shape = si.Shape(batch=16, seqlen=1, nheads=8, headdim=64, dstate=128, ngroups=2)
    prm, pools = _setup(shape, 64)
    pool0 = pools["ssm_pool"].clone()
    cpool0 = pools["conv_pool"].clone()
    slots = pools["slot_ids"]
    steps = 8
    ins = [_inputs(shape, t) for t in range(steps)]
    ys = [_step(shape, prm, pools, ins[t]) for t in range(steps)]
    # (i) slots not in slot_ids are byte-identical
    mask = torch.ones(64, dtype=torch.bool, device="cuda")
    mask[slots.long()] = False
    assert torch.equal(pools["ssm_pool"][mask], pool0[mask])
    assert torch.equal(pools["conv_pool"][mask], cpool0[mask])
    # (ii) the same sequences in permuted rows give byte-identical results
    perm = torch.randperm(16, generator=torch.Generator().manual_seed(9)).cuda()
    pool_b, cpool_b = pool0.clone(), cpool0.clone()
    ys_b = []
    for t in range(steps):
        inp = {k: v[perm].contiguous() for k, v in ins[t].items()}
        ys_b.append(_step(shape, prm, pools, inp, slots=slots[perm].contiguous(), pool=pool_b,
                          conv_pool=cpool_b))
    for t in range(steps):
        assert torch.equal(ys_b[t], ys[t][perm])
    assert torch.equal(pool_b, pools["ssm_pool"])
    assert torch.equal(cpool_b, pools["conv_pool"])
    # (iii) in place at the slots == a gathered contiguous copy, identity slots
    g_pool = pool0[slots.long()].contiguous()
    g_cpool = cpool0[slots.long()].contiguous()
    ident = torch.arange(16, dtype=torch.int32, device="cuda")
    for t in range(steps):
        yg = _step(shape, prm, pools, ins[t], slots=ident, pool=g_pool, conv_pool=g_cpool)
        assert torch.equal(yg, ys[t])
    assert torch.equal(g_pool, pools["ssm_pool"][slots.long()])
    assert torch.equal(g_cpool, pools["conv_pool"][slots.long()])


def test_bad_slot_sets_error_word_and_writes_nothing():
    shape = si.Shape(batch=4, seqlen=1, nheads=4, headdim=64, dstate=128, ngroups=1)
    prm, pools = _setup(shape, 8)
    assert ssd.ssd_read_device_error() == ssd.SSD_OK
    slots = torch.tensor([2, 8, 5, -1], dtype=torch.int32, device="cuda")
    pool0 = pools["ssm_pool"].clone()
    cpool0 = pools["conv_pool"].clone()
    inp = _inputs(shape, 0)
    y = _step(shape, prm, pools, inp, slots=slots)
    assert ssd.ssd_read_device_error() == ssd.SSD_ERR_BAD_SLOT
    assert ssd.ssd_read_device_error() == ssd.SSD_OK  # read clears it
    changed = [bool((pools["ssm_pool"][s] != pool0[s]).any()) for s in range(8)]
    assert changed == [s in (2, 5) for s in range(8)]
    cchanged = [bool((pools["conv_pool"][s] != cpool0[s]).any()) for s in range(8)]
    assert cchanged == [s in (2, 5) for s in range(8)]
    assert torch.isfinite(y[0].float()).all() and torch.isfinite(y[2].float()).all()


def test_decode_full_size_every_row():
    """256 rows in a 1024-slot pool [1024,128,64,128] fp32, 64 steps: every y of
    every row and step, every touched slot's SSM state (tolerance) and conv
    state (bit for bit) against the oracle, which follows each row through the
    64 steps as one 64-row sequence from the slot's initial states.  Untouched
    slots stay bit-identical."""
    shape = si.DECODE
    prm, pools = _setup(shape, si.DECODE_SLOTS)
    sl = pools["slot_ids"].long()
    h0_all = pools["ssm_pool"][sl].clone()
    c0_all = pools["conv_pool"][sl].clone()
    untouched = torch.ones(si.DECODE_SLOTS, dtype=torch.bool, device="cuda")
    untouched[sl] = False
    probe = torch.nonzero(untouched).flatten()[:64]
    pool_probe = pools["ssm_pool"][probe].clone()
    cpool_probe = pools["conv_pool"][probe].clone()
    xs, dts, zs, ys = [], [], [], []
    for t in range(si.DECODE_STEPS):
        inp = _inputs(shape, t)
        ys.append(_step(shape, prm, pools, inp))
        xs.append(inp["xbc"])
        dts.append(inp["dt_raw"])
        zs.append(inp["z"])
    X, DT, Z, Y = (torch.stack(v, 1) for v in (xs, dts, zs, ys))  # [R, steps, ...]
    assert torch.equal(pools["ssm_pool"][probe], pool_probe)
    assert torch.equal(pools["conv_pool"][probe], cpool_probe)
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    R = si.DECODE_ROWS
    ey, eh = MaxRel("y"), MaxRel("pool")
    for r0 in range(0, R, 32):
        rr = slice(r0, r0 + 32)
        y_o, h_o, c_o = oracle.mixer_prefill(
            f64(X[rr]), f64(prm["conv_w"]), f64(DT[rr]), f64(prm["A"]), H=H, P=P, N=N, G=G,
            conv_b=f64(prm["conv_b"]), conv_state=f64(c0_all[rr]), dt_bias=f64(prm["dt_bias"]),
            D=f64(prm["D"]), z=f64(Z[rr]), h0=f64(h0_all[rr]))
        ey.add(Y[rr], y_o)
        eh.add(pools["ssm_pool"][sl[rr]], h_o)
        assert np.array_equal(f64(pools["conv_pool"][sl[rr]]), c_o)
    ey.check(TOL[torch.bfloat16], R * si.DECODE_STEPS * H * P)
    eh.check(TOL[torch.bfloat16], R * H * P * N)


# ---------------------------------------------------------------------------
# K tokens per row in one call (multi-token decode): the state read once,
# stepped K times, written once

def _multi_inputs(shape, K, seed, act):
    g = torch.Generator().manual_seed(seed)
    R, H, P, C = shape.batch, shape.nheads, shape.headdim, shape.cdim
    return {"xbc": torch.randn((R, K, C), generator=g).to(act).cuda(),
            "dt_raw": torch.randn((R, K, H), generator=g).cuda(),
            "z": torch.randn((R, K, H * P), generator=g).to(act).cuda()}


def _multi_step(shape, prm, inp, slots, pool, cpool, conv=True, K=None):
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    R = inp["xbc"].shape[0]
    K = inp["xbc"].shape[1] if K is None else K
    d = ssd.dims(R, K, H, P, N, G, shape.conv_width)
    y = torch.full((R, K, H, P), float("nan"), dtype=inp["xbc"].dtype, device="cuda")
    ssd.ssd_decode_step(d, ssd.act_of(inp["xbc"]), ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z,
                        inp["xbc"], prm["conv_w"] if conv else None,
                        prm["conv_b"] if conv else None, cpool if conv else None, inp["dt_raw"],
                        prm["dt_bias"], prm["A"], prm["D"], inp["z"], slots, pool.shape[0], pool, y)
    return y


@pytest.mark.parametrize("K", [2, 3, 4, 7, 16])
@pytest.mark.parametrize("act,conv", [(torch.bfloat16, True), (torch.float32, True),
                                      (torch.bfloat16, False)])
def test_multi_token_decode_equals_single_steps_and_oracle(K, act, conv):
    """One call with K tokens per row == K calls of one token, bit for bit
    (the same arithmetic, the state kept in registers between the tokens
    instead of in the pool), and == the oracle's K steps from the slots'
    states, within the tolerance; slots no row names stay untouched."""
    shape = si.Shape(batch=12, seqlen=1, nheads=8, headdim=64, dstate=128, ngroups=2)
    _check_multi_token(shape, K, act, conv)


@pytest.mark.parametrize("K", [2, 16])
def test_multi_token_decode_wide_group(K):
    """32 heads in one group: at K = 16 the tokens' SiLU(z) no longer fits in
    shared memory beside their x columns and the kernel reads z in its
    epilogue instead (at K = 2 it stages it); either way the same results as
    K one-token calls, bit for bit, and as the oracle within the tolerance."""
    shape = si.Shape(batch=6, seqlen=1, nheads=32, headdim=64, dstate=128, ngroups=1)
    _check_multi_token(shape, K, torch.bfloat16, True)


def _check_multi_token(shape, K, act, conv):
    prm, pools = _setup(shape, 40, act=act)
    slots = pools["slot_ids"]
    inp = _multi_inputs(shape, K, seed=K, act=act)
    pool0, cpool0 = pools["ssm_pool"].clone(), pools["conv_pool"].clone()
    pa, ca = pool0.clone(), cpool0.clone()
    y = _multi_step(shape, prm, inp, slots, pa, ca, conv=conv)
    pb, cb = pool0.clone(), cpool0.clone()
    ys = []
    for t in range(K):
        one = {k: v[:, t:t + 1].contiguous() for k, v in inp.items()}
        ys.append(_multi_step(shape, prm, one, slots, pb, cb, conv=conv))
    assert torch.equal(y, torch.cat(ys, dim=1))
    assert torch.equal(pa, pb) and torch.equal(ca, cb)
    sl = slots.long()
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    y_o, h_o, c_o = oracle.mixer_prefill(
        f64(inp["xbc"]), f64(prm["conv_w"]) if conv else None, f64(inp["dt_raw"]),
        f64(prm["A"]), H=H, P=P, N=N, G=G, conv_b=f64(prm["conv_b"]) if conv else None,
        conv_state=f64(cpool0[sl]) if conv else None, dt_bias=f64(prm["dt_bias"]),
        D=f64(prm["D"]), z=f64(inp["z"]), h0=f64(pool0[sl]))
    R = shape.batch
    assert_close(y, y_o, TOL[act], count=R * K * H * P, what="y")
    assert_close(pa[sl], h_o, TOL[act], count=R * H * P * N, what="pool")
    if conv:
        assert np.array_equal(f64(ca[sl]), c_o)
    untouched = [s for s in range(40) if s not in set(slots.tolist())]
    assert torch.equal(pa[untouched], pool0[untouched])
    assert torch.equal(ca[untouched], cpool0[untouched])


def test_multi_token_decode_bad_slot_and_token_limit():
    shape = si.Shape(batch=3, seqlen=1, nheads=4, headdim=64, dstate=128, ngroups=1)
    prm, pools = _setup(shape, 8)
    slots = torch.tensor([1, 9, 4], dtype=torch.int32, device="cuda")
    pool0, cpool0 = pools["ssm_pool"].clone(), pools["conv_pool"].clone()
    inp = _multi_inputs(shape, 5, seed=2, act=torch.bfloat16)
    assert ssd.ssd_read_device_error() == ssd.SSD_OK
    _multi_step(shape, prm, inp, slots, pools["ssm_pool"], pools["conv_pool"])
    assert ssd.ssd_read_device_error() == ssd.SSD_ERR_BAD_SLOT
    changed = [bool((pools["ssm_pool"][s] != pool0[s]).any()) for s in range(8)]
    assert changed == [s in (1, 4) for s in range(8)]
    inp17 = _multi_inputs(shape, 17, seed=3, act=torch.bfloat16)
    with pytest.raises(ssd.SsdError) as e:
        _multi_step(shape, prm, inp17, slots, pools["ssm_pool"], pools["conv_pool"])
    assert e.value.status == ssd.SSD_ERR_UNSUPPORTED
