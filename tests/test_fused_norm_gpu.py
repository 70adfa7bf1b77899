"""GPU parity of ssd_chunk_scan_gated_norm -- the scan, then the gated group
RMSNorm over its output, in one call (TensorSharp "nemotron.md" section 3:
out = SiLU(z) * GroupRMSNorm(y, ssm_norm.weight); section 4.1: y normalised
per group before the gate) -- against the oracle's scan without the gate
followed by the oracle's norm, on the same stored inputs; tolerance as in
tests/helpers.py."""
import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
from tests.helpers import (TOL, MaxRel, assert_close, f64, make_problem, oracle_prefill,
                           oracle_prefill_by_group)

pytestmark = pytest.mark.gpu

ssd = pytest.importorskip("ssd_scan_gb300")

EPS = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ssd.load_library()
    yield
    assert ssd.ssd_read_device_error() == ssd.SSD_OK


def _weights(C, seed=2):
    return torch.rand((C,), generator=torch.Generator().manual_seed(seed)) + 0.5


def _fused(shape, dev, w, splits, conv=True):
    """ssd_chunk_scan_gated_norm over the rows, one call per split, chaining
    the states.  Returns (y [B,S,H,P], ssm state, conv state)."""
    B, S = shape.batch, shape.seqlen
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    xbc = dev["xbc"]
    y = torch.empty((B, S, H, P), dtype=xbc.dtype, device=xbc.device)
    h, cs = dev["ssm_state"], dev["conv_state"] if conv else None
    r0 = 0
    for L in splits:
        ys, h, cs = ssd.chunk_scan(
            xbc[:, r0:r0 + L].contiguous(), dev["dt_raw"][:, r0:r0 + L].contiguous(), dev["A"],
            nheads=H, headdim=P, dstate=N, ngroups=G,
            conv_w=dev["conv_w"] if conv else None, conv_b=dev["conv_b"] if conv else None,
            conv_state=cs, dt_bias=dev["dt_bias"], D=dev["D"],
            z=dev["z"][:, r0:r0 + L].contiguous(), ssm_state=h, norm_w=w, norm_eps=EPS)
        y[:, r0:r0 + L] = ys
        r0 += L
    return y, h, cs


def _plain(shape, dev, splits, conv=True):
    """The same rows through ssd_chunk_scan without the gate."""
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    ys, h, cs = [], dev["ssm_state"], dev["conv_state"] if conv else None
    r0 = 0
    for L in splits:
        y, h, cs = ssd.chunk_scan(
            dev["xbc"][:, r0:r0 + L].contiguous(), dev["dt_raw"][:, r0:r0 + L].contiguous(),
            dev["A"], nheads=H, headdim=P, dstate=N, ngroups=G,
            conv_w=dev["conv_w"] if conv else None, conv_b=dev["conv_b"] if conv else None,
            conv_state=cs, dt_bias=dev["dt_bias"], D=dev["D"], z=None, ssm_state=h)
        ys.append(y)
        r0 += L
    return torch.cat(ys, dim=1), h, cs


def _oracle(shape, cpu, w, conv=True):
    no_z = {k: v for k, v in cpu.items() if k != "z"}
    yo, hS, cso, _ = oracle_prefill(shape, no_z, conv=conv)
    B, S, H, P = yo.shape
    ref = oracle.gated_group_rmsnorm(yo.reshape(B, S, H * P), f64(cpu["z"]), f64(w), EPS,
                                     shape.ngroups)
    return ref.reshape(B, S, H, P), hS, cso


# 300 rows: two full chunks and a ragged one; split in two calls, each ragged;
# 137 rows of one sequence: an odd row count (the scale pass's last block
# holds one row)
@pytest.mark.parametrize("B,S,splits", [(2, 300, [300]), (2, 300, [170, 130]),
                                        (1, 137, [137])])
@pytest.mark.parametrize("conv", [True, False])
def test_fused_gated_norm_matches_oracle(B, S, splits, conv):
    shape = si.Shape(batch=B, seqlen=S, nheads=8, headdim=64, dstate=128, ngroups=2)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=11, with_z=True)
    w = _weights(shape.nheads * shape.headdim)
    before = ssd.ssd_launch_counts()
    y, h, cs = _fused(shape, dev, w.cuda(), splits, conv=conv)
    after = ssd.ssd_launch_counts()
    # the tensor-core scan and the scale pass, once per call; no separate norm
    assert after["scan_tc"] - before["scan_tc"] == len(splits)
    assert after["norm_scale"] - before["norm_scale"] == len(splits)
    assert after["gated_norm"] == before["gated_norm"]
    ref, hS, cso = _oracle(shape, cpu, w, conv=conv)
    assert_close(y, ref, TOL[torch.bfloat16], count=y.numel(), what="fused scan + gated norm")
    assert_close(h, hS, TOL[torch.bfloat16], count=h.numel(), what="ssm state")
    # the states do not depend on the norm: bit for bit those of the plain scan
    y0, h0, cs0 = _plain(shape, dev, splits, conv=conv)
    assert torch.equal(h, h0)
    if conv:
        assert torch.equal(cs, cs0)
    # and the two-kernel composition agrees with the fused call
    y2 = ssd.gated_group_rmsnorm(y0.reshape(B, S, -1), dev["z"], w.cuda(),
                                 ngroups=shape.ngroups, eps=EPS)
    assert_close(y, f64(y2).reshape(y.shape), TOL[torch.bfloat16], count=y.numel(),
                 what="fused against scan, then norm")


@pytest.mark.parametrize("act,S,P", [(torch.float32, 37, 64), (torch.bfloat16, 3, 32)])
def test_fused_gated_norm_on_the_row_exact_kernel(act, S, P):
    """fp32, and bf16 heads of 32 channels (not the tensor-core shape): the
    scan without the gate, then the norm in place, behind the same call."""
    shape = si.Shape(batch=2, seqlen=S, nheads=8, headdim=P, dstate=128, ngroups=2)
    cpu, dev = make_problem(shape, act=act, seed=4, with_z=True)
    w = _weights(shape.nheads * shape.headdim, seed=6)
    before = ssd.ssd_launch_counts()
    y, h, _ = _fused(shape, dev, w.cuda(), [S])
    after = ssd.ssd_launch_counts()
    assert after["scan_simt"] - before["scan_simt"] == 1
    assert after["gated_norm"] - before["gated_norm"] == 1
    assert after["norm_scale"] == before["norm_scale"]
    ref, hS, _ = _oracle(shape, cpu, w)
    assert_close(y, ref, TOL[act], count=y.numel(), what="row-exact scan + gated norm")
    assert_close(h, hS, TOL[act], count=h.numel(), what="ssm state")


def test_fused_gated_norm_groups_of_three_heads_take_the_two_kernel_path():
    """Norm groups of 3 heads (192 channels) do not split into the scale
    pass's 256-channel warp blocks: the scan without the gate, then the norm."""
    shape = si.Shape(batch=2, seqlen=150, nheads=6, headdim=64, dstate=128, ngroups=2)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=5, with_z=True)
    w = _weights(shape.nheads * shape.headdim, seed=9)
    before = ssd.ssd_launch_counts()
    y, h, _ = _fused(shape, dev, w.cuda(), [150])
    after = ssd.ssd_launch_counts()
    assert after["scan_tc"] - before["scan_tc"] == 1
    assert after["gated_norm"] - before["gated_norm"] == 1
    assert after["norm_scale"] == before["norm_scale"]
    ref, hS, _ = _oracle(shape, cpu, w)
    assert_close(y, ref, TOL[torch.bfloat16], count=y.numel(), what="scan + gated norm")
    assert_close(h, hS, TOL[torch.bfloat16], count=h.numel(), what="ssm state")


def test_fused_gated_norm_full_size_every_element():
    """The Nemotron-H-8B mixer at 2048 rows (128 heads, 8 groups of 16 heads =
    1024 channels per norm group): every element of y against the oracle,
    one group at a time (a norm group is an SSM group's heads)."""
    shape = si.PREFILL
    H, P, G = shape.nheads, shape.headdim, shape.ngroups
    hpg = H // G
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=21, with_z=True)
    w = _weights(H * P, seed=8)
    y, h, _ = _fused(shape, dev, w.cuda(), [shape.seqlen])
    no_z = {k: v for k, v in cpu.items() if k != "z"}
    ey, eh = MaxRel("y"), MaxRel("ssm_state")
    for b in range(shape.batch):
        for g in range(G):
            heads, yo, ho, _, _ = oracle_prefill_by_group(shape, no_z, b, g)
            cols = slice(g * hpg * P, (g + 1) * hpg * P)
            ref = oracle.gated_group_rmsnorm(yo.reshape(1, shape.seqlen, hpg * P),
                                             f64(cpu["z"][b][:, cols])[None],
                                             f64(w[cols]), EPS, 1)
            ey.add(y[b, :, int(heads[0]):int(heads[-1]) + 1], ref.reshape(yo.shape))
            eh.add(h[b, int(heads[0]):int(heads[-1]) + 1], ho)
    ey.check(TOL[torch.bfloat16], shape.batch * shape.seqlen * H * P)
    eh.check(TOL[torch.bfloat16], shape.batch * H * P * shape.dstate)


def test_fused_gated_norm_rejects_bad_arguments_without_launching():
    shape = si.Shape(batch=1, seqlen=130, nheads=8, headdim=64, dstate=128, ngroups=2)
    _, dev = make_problem(shape, act=torch.bfloat16, seed=1, with_z=True)
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    d = ssd.dims(1, 130, H, P, N, G, 4, 128)
    act, f = ssd.SSD_BF16, ssd.SSD_DT_SOFTPLUS
    w = _weights(H * P).cuda()
    y = torch.empty((1, 130, H, P), dtype=torch.bfloat16, device="cuda")
    hs = torch.empty((1, H, P, N), dtype=torch.float32, device="cuda")
    cs = torch.empty_like(dev["conv_state"])
    need = ssd.ssd_chunk_scan_workspace_size(d, act, f | ssd.SSD_GATED_NORM, True)
    plain = ssd.ssd_chunk_scan_workspace_size(d, act, f, True)
    assert need == plain + 8 * 130 * 4 + 256 - (8 * 130 * 4) % 256  # + the [B,H,S] sums
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def call(z=dev["z"], w=w, eps=EPS, ws=ws, flags=f):
        ssd.ssd_chunk_scan_gated_norm(d, act, flags, dev["xbc"], dev["conv_w"], dev["conv_b"],
                                      dev["conv_state"], cs, dev["dt_raw"], dev["dt_bias"],
                                      dev["A"], dev["D"], z, w, eps, dev["ssm_state"], y, hs, ws)

    before = ssd.ssd_launch_counts()
    for kw, status in [(dict(w=None), ssd.SSD_ERR_INVALID_ARG),
                       (dict(z=None), ssd.SSD_ERR_INVALID_ARG),
                       (dict(eps=float("nan")), ssd.SSD_ERR_INVALID_ARG),
                       (dict(eps=-1.0), ssd.SSD_ERR_INVALID_ARG),
                       (dict(ws=ws[:plain]), ssd.SSD_ERR_INVALID_ARG),
                       (dict(flags=f | 8), ssd.SSD_ERR_INVALID_ARG)]:
        with pytest.raises(ssd.SsdError) as e:
            call(**kw)
        assert e.value.status == status, kw
    assert ssd.ssd_launch_counts() == before
    # SSD_HAS_Z and SSD_GATED_NORM are implied and accepted
    call(flags=f | ssd.SSD_HAS_Z | ssd.SSD_GATED_NORM)
    assert ssd.ssd_read_device_error() == ssd.SSD_OK
    assert np.all(np.isfinite(f64(y)))
