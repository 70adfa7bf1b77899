"""Sequence-parallel state passing over ranks on CPU: two and three gloo ranks
on 127.0.0.1 drive ssd_scan_gb300.seqpar.sequence_parallel_scan, each rank
holding one consecutive segment of the rows.  The per-rank steps are the fp64
oracle's (conv + recurrence, segment decay, state combine), so what is tested
here is the exchange: the conv halos, the all-gather of (Gamma_k, h_k), the
chain in rank order and the second pass.  Each rank's rows of y, and the
final states, must equal one oracle call over all rows."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _problem():
    import ssd_inputs as si
    shape = si.TINY.with_(batch=2, seqlen=13)
    prm = si.params(shape, seed=7)
    inp = si.prefill_inputs(shape, seed=7, act_dtype=torch.float64, with_z=True)
    return shape, {**prm, **inp}


def _oracle_ops(shape, p):
    import oracle
    from ssd_scan_gb300.seqpar import SegmentOps
    f = lambda t: None if t is None else t.detach().to(torch.float64).numpy()  # noqa: E731
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups

    def scan(xbc, dt, z, h0, conv_state):
        y, h, cs = oracle.mixer_prefill(f(xbc), f(p["conv_w"]), f(dt), f(p["A"]), H=H, P=P, N=N,
                                        G=G, conv_b=f(p["conv_b"]), conv_state=f(conv_state),
                                        dt_bias=f(p["dt_bias"]), D=f(p["D"]), z=f(z), h0=f(h0))
        return torch.from_numpy(y), torch.from_numpy(h), torch.from_numpy(cs)

    def decay(dt):
        return torch.from_numpy(oracle.segment_decay(f(dt), f(p["A"]), dt_bias=f(p["dt_bias"])))

    def combine(g, h_prev, h_seg):
        return torch.from_numpy(oracle.state_combine(f(g), f(h_prev), f(h_seg)))

    return SegmentOps(scan, decay, combine)


def _worker(rank, world, port, cuts, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from ssd_scan_gb300.seqpar import sequence_parallel_scan
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shape, p = _problem()
        edges = [0] + cuts + [shape.seqlen]
        a, b = edges[rank], edges[rank + 1]
        seg = {k: p[k][:, a:b].contiguous() for k in ("xbc", "dt_raw", "z")}
        y, h, cs = sequence_parallel_scan(_oracle_ops(shape, p), seg["xbc"], seg["dt_raw"],
                                          seg["z"], p["ssm_state"], p["conv_state"],
                                          conv_width=shape.conv_width)
        out[rank] = (y.numpy(), h.numpy(), cs.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("cuts", [[6], [4, 9]])
def test_gloo_ranks_equal_one_call(cuts):
    import oracle
    world = len(cuts) + 1
    port = _free_port()
    out = mp.Manager().dict()
    mp.start_processes(_worker, args=(world, port, cuts, out), nprocs=world, start_method="spawn")
    shape, p = _problem()
    f = lambda t: t.detach().numpy()  # noqa: E731
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    y, h, cs = oracle.mixer_prefill(f(p["xbc"]), f(p["conv_w"]), f(p["dt_raw"]), f(p["A"]), H=H,
                                    P=P, N=N, G=G, conv_b=f(p["conv_b"]),
                                    conv_state=f(p["conv_state"]), dt_bias=f(p["dt_bias"]),
                                    D=f(p["D"]), z=f(p["z"]), h0=f(p["ssm_state"]))
    edges = [0] + cuts + [shape.seqlen]
    ys = np.concatenate([out[r][0] for r in range(world)], axis=1)
    assert ys.shape == y.shape
    den = np.abs(y).max()
    assert np.abs(ys - y).max() / den < 1e-12
    for r in range(world):
        assert np.abs(out[r][1] - h).max() / np.abs(h).max() < 1e-12
        assert np.array_equal(out[r][2], cs)
    assert edges[-1] == shape.seqlen


def test_segment_too_short_for_the_conv_halo_is_refused():
    from ssd_scan_gb300.seqpar import halo_rows
    with pytest.raises(ValueError):
        halo_rows(torch.zeros(1, 2, 8), 4)
