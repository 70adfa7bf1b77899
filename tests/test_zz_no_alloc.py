"""ssd_chunk_scan_static_ws, the entry point for callers that cannot allocate
device memory (a plugin inside a host program that owns the device pool, or a
serving loop that keeps cudaMalloc off its hot path).  It takes its scratch
from the library's fixed per-GPU array instead of a caller workspace.

These tests call it through the C-ABI and compare it with ssd_chunk_scan
given a workspace of its own, on two calls in a row: the second call runs a
different, smaller problem over an array that still holds the first call's
rows, so a result that leaned on stale or zeroed scratch would show.  The
file is named to be collected last.
"""
import pytest
import torch

import ssd_inputs as si
from tests.helpers import TOL, assert_close, make_problem

pytestmark = pytest.mark.gpu

ssd = pytest.importorskip("ssd_scan_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ssd.load_library()
    yield
    assert ssd.ssd_read_device_error() == ssd.SSD_OK


def _outputs(shape, dev):
    B, S, H, P, N, W = (shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                        shape.conv_width)
    xbc = dev["xbc"]
    y = torch.full((B, S, H, P), float("nan"), dtype=xbc.dtype, device=xbc.device)
    h = torch.full((B, H, P, N), float("nan"), dtype=torch.float32, device=xbc.device)
    cs = torch.full((B, W - 1, shape.cdim), float("nan"), dtype=xbc.dtype, device=xbc.device)
    return y, h, cs


def _args(dev, out):
    y, h, cs = out
    return (dev["xbc"], dev["conv_w"], dev["conv_b"], dev["conv_state"], cs, dev["dt_raw"],
            dev["dt_bias"], dev["A"], dev["D"], dev["z"], dev["ssm_state"], y, h)


def _run_both(shape, seed):
    """One problem through both entry points; returns (static_ws, workspace) outputs."""
    cpu, dev = make_problem(shape, seed=seed, act=torch.bfloat16)
    d = ssd.dims(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                 shape.ngroups, shape.conv_width, shape.chunk)
    flags = ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z
    need = ssd.ssd_chunk_scan_workspace_size(d, ssd.SSD_BF16, flags, True)
    assert 0 < need <= ssd.SSD_STATIC_SCRATCH_BYTES
    before = ssd.ssd_launch_counts()
    got = _outputs(shape, dev)
    ssd.ssd_chunk_scan_static_ws(d, ssd.SSD_BF16, flags, *_args(dev, got))
    after = ssd.ssd_launch_counts()
    # the scratch-using path ran: the B|C conv wrote the scratch, the scan read it
    assert after["bc_conv"] - before["bc_conv"] == 1
    assert after["scan_tc"] - before["scan_tc"] == 1
    ref = _outputs(shape, dev)
    ws = ssd.workspace_for(d, ssd.SSD_BF16, flags, True, dev["xbc"].device)
    ssd.ssd_chunk_scan(d, ssd.SSD_BF16, flags, *_args(dev, ref), workspace=ws)
    torch.cuda.synchronize()
    return got, ref


def _compare(shape, got, ref):
    """Both entry points run the same kernels on the same inputs, so every
    output must agree bit for bit (a stale scratch row that moved a few values
    within the tolerance would still show); the tolerance check is kept as the
    bound the other parity tests use."""
    tol = TOL[torch.bfloat16]
    B, S, H, P, N = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate
    assert_close(got[0], ref[0].float().cpu().double().numpy(), tol, count=B * S * H * P,
                 what="y")
    assert_close(got[1], ref[1].cpu().double().numpy(), tol, count=B * H * P * N,
                 what="ssm_state")
    assert torch.equal(got[0], ref[0]), "y must equal the workspace entry's, bit for bit"
    assert torch.equal(got[1], ref[1]), "ssm state must equal the workspace entry's"
    assert torch.equal(got[2], ref[2]), "conv state must be the raw rows, bit for bit"


def test_static_scratch_matches_workspace_entry_two_calls_in_a_row():
    first = si.Shape(batch=2, seqlen=600, nheads=8, headdim=64, dstate=128, ngroups=2)
    second = si.Shape(batch=1, seqlen=300, nheads=4, headdim=64, dstate=128, ngroups=1)
    got, ref = _run_both(first, seed=11)
    _compare(first, got, ref)
    got, ref = _run_both(second, seed=12)
    _compare(second, got, ref)


def test_static_scratch_rejects_problems_larger_than_the_array():
    # B|C scratch of 33024 rows x 2 x 128 bf16 = 16.1 MiB > 16 MiB
    shape = si.Shape(batch=1, seqlen=33024, nheads=2, headdim=64, dstate=128, ngroups=1)
    d = ssd.dims(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                 shape.ngroups, shape.conv_width, shape.chunk)
    flags = ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z
    assert ssd.ssd_chunk_scan_workspace_size(d, ssd.SSD_BF16, flags, True) > \
        ssd.SSD_STATIC_SCRATCH_BYTES
    _, dev = make_problem(shape, seed=3, act=torch.bfloat16)
    out = _outputs(shape, dev)
    before = ssd.ssd_launch_counts()
    with pytest.raises(ssd.SsdError) as e:
        ssd.ssd_chunk_scan_static_ws(d, ssd.SSD_BF16, flags, *_args(dev, out))
    assert e.value.status == ssd.SSD_ERR_UNSUPPORTED
    assert ssd.ssd_launch_counts() == before, "a rejected call must launch nothing"
    assert torch.isnan(out[0]).all()


def test_static_scratch_size_check_comes_before_the_argument_checks():
    """A problem too large for the array is refused as unsupported before any
    other argument is looked at: even with a null y it returns
    SSD_ERR_UNSUPPORTED (ssd_chunk_scan itself would say invalid argument)."""
    shape = si.Shape(batch=1, seqlen=33024, nheads=2, headdim=64, dstate=128, ngroups=1)
    d = ssd.dims(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                 shape.ngroups, shape.conv_width, shape.chunk)
    flags = ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z
    _, dev = make_problem(shape, seed=3, act=torch.bfloat16)
    y, h, cs = _outputs(shape, dev)
    args = list(_args(dev, (y, h, cs)))
    args[11] = None  # y
    with pytest.raises(ssd.SsdError) as e:
        ssd.ssd_chunk_scan_static_ws(d, ssd.SSD_BF16, flags, *args)
    assert e.value.status == ssd.SSD_ERR_UNSUPPORTED
