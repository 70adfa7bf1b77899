"""GPU parity of sequence-parallel state passing: ssd_segment_decay and
ssd_state_combine against the fp64 oracle, and a 2048-row prefill split into
K segments scanned as K ranks would (conv halos, pass 1 from a zero state,
the chain of (Gamma_k, h_k), pass 2), run one after another on this GPU with
the library's own steps: every element of y and the final state against the
oracle, as for one call."""
import numpy as np
import pytest
import torch

import oracle
import ssd_inputs as si
from tests.helpers import TOL, assert_close, check_prefill_every_element, f64, make_problem

pytestmark = pytest.mark.gpu

ssd = pytest.importorskip("ssd_scan_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ssd.load_library()
    yield
    assert ssd.ssd_read_device_error() == ssd.SSD_OK


@pytest.mark.parametrize("stress,S", [(False, 2048), (True, 4096), (False, 1), (False, 0)])
def test_segment_decay_matches_oracle(stress, S):
    shape = (si.STRESS if stress else si.PREFILL).with_(batch=3, seqlen=S)
    prm = {k: v.cuda() for k, v in si.params(shape, seed=5, stress=stress).items()}
    dt = si.prefill_inputs(shape, seed=5, device="cuda", stress=stress)["dt_raw"]
    g = torch.full((3, shape.nheads), float("nan"), device="cuda")
    c0 = ssd.ssd_launch_counts()["segment_decay"]
    ssd.ssd_segment_decay(ssd.dims(3, S, shape.nheads, 64, 128, 8), ssd.SSD_DT_SOFTPLUS, dt,
                          prm["dt_bias"], prm["A"], g)
    torch.cuda.synchronize()
    assert ssd.ssd_launch_counts()["segment_decay"] == c0 + 1
    go = oracle.segment_decay(f64(dt), f64(prm["A"]), dt_bias=f64(prm["dt_bias"]))
    if S == 0:
        assert torch.equal(g, torch.zeros_like(g))
    else:
        assert_close(g, go, 1e-6, count=3 * shape.nheads, what="gamma")


@pytest.mark.parametrize("with_prev", [True, False])
@pytest.mark.parametrize("in_place", [False, True])
def test_state_combine_matches_oracle(with_prev, in_place):
    g_ = torch.Generator(device="cuda").manual_seed(3)
    B, H, P, N = 2, 16, 64, 128
    gamma = -torch.rand((B, H), generator=g_, device="cuda") * 8.0
    gamma[0, 0] = 0.5  # a rising total: the clamp keeps exp(min(Gamma, 0)) = 1
    hp = torch.randn((B, H, P, N), generator=g_, device="cuda")
    hs = torch.randn((B, H, P, N), generator=g_, device="cuda")
    ho = oracle.state_combine(f64(gamma), f64(hp) if with_prev else None, f64(hs))
    out = hs if in_place else torch.empty_like(hs)
    ssd.ssd_state_combine(ssd.dims(B, 0, H, P, N, 1), gamma, hp if with_prev else None, hs, out)
    assert_close(out, ho, 1e-6, count=B * H * P * N, what="combined state")


@pytest.mark.parametrize("K", [2, 4])
def test_segments_as_ranks_equal_one_call(K):
    from ssd_scan_gb300.seqpar import chain, cuda_ops, halo_rows, pass1
    shape = si.PREFILL
    cpu, dev = make_problem(shape, act=torch.bfloat16, seed=21)
    H, P, N, G, W = shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.conv_width
    ops = cuda_ops(dev["A"], nheads=H, headdim=P, dstate=N, ngroups=G, conv_w=dev["conv_w"],
                   conv_b=dev["conv_b"], dt_bias=dev["dt_bias"], D=dev["D"])
    L = shape.seqlen // K
    segs = [{k: dev[k][:, i * L:(i + 1) * L].contiguous() for k in ("xbc", "dt_raw", "z")}
            for i in range(K)]
    cs_in = [dev["conv_state"]] + [halo_rows(segs[i]["xbc"], W) for i in range(K - 1)]
    gs, hs = zip(*[pass1(ops, s["xbc"], s["dt_raw"], s["z"], c) for s, c in zip(segs, cs_in)])
    h_in = chain(ops, gs, hs, dev["ssm_state"])
    ys = [ops.scan(s["xbc"], s["dt_raw"], s["z"], h, c)[0] for s, c, h in zip(segs, cs_in, h_in)]
    y = torch.cat(ys, dim=1)
    cs = halo_rows(segs[-1]["xbc"], W)
    check_prefill_every_element(shape, cpu, y, h_in[K], cs, torch.bfloat16)
