"""GPU parity of the gated group RMSNorm (group RMSNorm of y, then the SiLU(z)
gate; TensorSharp "nemotron.md" sections 3, 4.1, 6) through the C-ABI, against
the fp64 oracle on the same stored inputs; tolerance as in tests/helpers.py."""
import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
from tests.helpers import TOL, assert_close, f64, gpu_prefill, make_problem, oracle_prefill

pytestmark = pytest.mark.gpu

ssd = pytest.importorskip("ssd_scan_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ssd.load_library()
    yield
    assert ssd.ssd_read_device_error() == ssd.SSD_OK


def _inputs(B, S, C, act, seed):
    g = torch.Generator().manual_seed(seed)
    y = (torch.randn((B, S, C), generator=g) * 2.0).to(act)
    z = torch.randn((B, S, C), generator=g).to(act)
    w = torch.rand((C,), generator=g) + 0.5
    return y, z, w


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("in_place", [False, True])
# groups of 256 and 2048 channels (one CTA a group) and of 136 (one warp a group)
@pytest.mark.parametrize("H,P,G", [(8, 64, 2), (32, 128, 2), (17, 8, 1)])
def test_gated_norm_matches_oracle(act, in_place, H, P, G):
    B, S = 2, 37
    C = H * P
    y, z, w = _inputs(B, S, C, act, seed=3)
    ref = oracle.gated_group_rmsnorm(f64(y), f64(z), f64(w), 1e-5, G)
    yd, zd, wd = y.cuda(), z.cuda(), w.cuda()
    before = ssd.ssd_launch_counts()["gated_norm"]
    out = ssd.gated_group_rmsnorm(yd, zd, wd, ngroups=G, eps=1e-5, out=yd if in_place else None)
    assert ssd.ssd_launch_counts()["gated_norm"] == before + 1
    if in_place:
        assert out.data_ptr() == yd.data_ptr()
    assert_close(out, ref, TOL[act], count=B * S * C, what="gated norm")


def test_gated_norm_full_size_every_row():
    """The Nemotron-H-8B mixer width: 8192 channels in 8 groups of 1024, 2048
    rows, bf16; every element against the oracle."""
    sh = si.PREFILL
    C, G = sh.nheads * sh.headdim, sh.ngroups
    y, z, w = _inputs(1, sh.seqlen, C, torch.bfloat16, seed=5)
    out = ssd.gated_group_rmsnorm(y.cuda(), z.cuda(), w.cuda(), ngroups=G, eps=1e-5)
    ref = oracle.gated_group_rmsnorm(f64(y), f64(z), f64(w), 1e-5, G)
    assert_close(out, ref, TOL[torch.bfloat16], count=sh.seqlen * C, what="gated norm")


def test_scan_then_gated_norm_matches_oracle_mixer():
    """The mixer's tail: the bf16 scan without the gate, then the gated group
    norm, against the oracle's scan followed by its norm."""
    shape = si.Shape(batch=2, seqlen=300, nheads=8, headdim=64, dstate=128, ngroups=2)
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=9, with_z=True)
    z = dev.pop("z")
    cpu_z = cpu.pop("z")
    y, _, _ = gpu_prefill(shape, dev, [180, 120])
    w = torch.rand((shape.nheads * shape.headdim,), generator=torch.Generator().manual_seed(2))
    out = ssd.gated_group_rmsnorm(y.reshape(2, 300, -1), z, w.cuda(), ngroups=shape.ngroups)
    yo, _, _, _ = oracle_prefill(shape, cpu)
    ref = oracle.gated_group_rmsnorm(yo.reshape(2, 300, -1), f64(cpu_z), f64(w), 1e-5,
                                     shape.ngroups)
    assert_close(out, ref, TOL[torch.bfloat16], count=y.numel(), what="scan + gated norm")


def test_gated_norm_rejects_bad_arguments_without_launching():
    y, z, w = (t.cuda() for t in _inputs(1, 4, 512, torch.bfloat16, seed=1))
    d = ssd.dims(1, 4, 8, 64, 1, 2)
    before = ssd.ssd_launch_counts()
    for eps in (float("nan"), -1.0, float("inf")):
        with pytest.raises(ssd.SsdError) as e:
            ssd.ssd_gated_group_rmsnorm(d, ssd.SSD_BF16, y, z, w, eps, y)
        assert e.value.status == ssd.SSD_ERR_INVALID_ARG
    with pytest.raises(ssd.SsdError) as e:  # out overlapping z
        ssd.ssd_gated_group_rmsnorm(d, ssd.SSD_BF16, y, z, w, 1e-5, z)
    assert e.value.status == ssd.SSD_ERR_INVALID_ARG
    with pytest.raises(ssd.SsdError) as e:  # groups of 4 channels: not whole 16-byte vectors
        ssd.ssd_gated_group_rmsnorm(ssd.dims(1, 4, 128, 4, 1, 128), ssd.SSD_BF16, y, z, w,
                                    1e-5, y)
    assert e.value.status == ssd.SSD_ERR_UNSUPPORTED
    assert ssd.ssd_launch_counts() == before
