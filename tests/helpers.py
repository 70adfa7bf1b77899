"""Glue for the parity tests: run the CUDA library and the fp64 oracle on the
same seeded inputs and compare them element by element.

Tolerance (per output tensor): max|gpu - oracle| / max|oracle| <= 1e-4 for fp32
activations and <= 2e-2 for bf16 activations; the oracle reads the exact
stored input values widened to fp64.  Every comparison also asserts the
element count against the geometry, so a comparison over nothing cannot pass.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import ssd_inputs as si

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def f64(t):
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(gpu, ref, count=None):
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if count is not None:
        assert g.size == count, (g.size, count)
    assert g.size > 0
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    den = float(np.max(np.abs(r)))
    err = float(np.max(np.abs(g - r)))
    return err / den if den > 0 else err


def assert_close(gpu, ref, tol, count=None, what=""):
    e = rel_err(gpu, ref, count)
    assert e <= tol, f"{what}: relative error {e:.3e} > {tol:.1e}"
    return e


def make_problem(shape: si.Shape, seed=0, act=torch.bfloat16, stress=False,
                 initial_state=True, with_z=True, device="cuda"):
    """Seeded inputs on the CPU, copied to the device.  Returns (cpu, dev)."""
    prm = si.params(shape, seed=seed, stress=stress)
    inp = si.prefill_inputs(shape, seed=seed, act_dtype=act, stress=stress,
                            initial_state=initial_state, with_z=with_z)
    cpu = {**prm, **inp}
    dev = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in cpu.items()}
    return cpu, dev


def gpu_prefill(shape: si.Shape, dev: dict, splits=None, conv=True, dt_softplus=True,
                act=None, stream=None):
    """Run ssd_chunk_scan over the rows, one call per entry of ``splits``
    (chaining the final states).  Returns (y, ssm_state, conv_state)."""
    import ssd_scan_gb300 as ssd
    B, S = shape.batch, shape.seqlen
    splits = splits or [S]
    assert sum(splits) == S
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    xbc = dev["xbc"]
    y = torch.empty((B, S, H, P), dtype=xbc.dtype, device=xbc.device)
    h = dev.get("ssm_state")
    cs = dev.get("conv_state") if conv else None
    r0 = 0
    for L in splits:
        xs = xbc[:, r0:r0 + L].contiguous()
        dts = dev["dt_raw"][:, r0:r0 + L].contiguous()
        zs = dev["z"][:, r0:r0 + L].contiguous() if dev.get("z") is not None else None
        ys, h, cs_new = ssd.chunk_scan(
            xs, dts, dev["A"], nheads=H, headdim=P, dstate=N, ngroups=G,
            conv_w=dev["conv_w"] if conv else None,
            conv_b=dev["conv_b"] if conv else None, conv_state=cs,
            dt_bias=dev["dt_bias"], D=dev["D"], z=zs, ssm_state=h,
            dt_softplus=dt_softplus, stream=stream)
        y[:, r0:r0 + L] = ys
        cs = cs_new
        r0 += L
    return y, h, cs


def oracle_prefill(shape: si.Shape, cpu: dict, conv=True, dt_softplus=True, heads=None,
                   batches=None, nthreads=None):
    """fp64 oracle of one prefill over all rows.  ``heads`` / ``batches``
    restrict it to a subset (each head then gets its own group's B/C columns,
    which the group-expansion pin shows leaves the result unchanged).
    Returns (y [b,S,h,P], hS [b,h,P,N], conv_state_out [b,W-1,cols] or None)."""
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    hpg = H // G
    heads = list(range(H)) if heads is None else list(heads)
    batches = list(range(shape.batch)) if batches is None else list(batches)
    cols = []
    for h in heads:
        cols += list(range(h * P, (h + 1) * P))
    for h in heads:
        g = h // hpg
        cols += list(range(H * P + g * N, H * P + (g + 1) * N))
    for h in heads:
        g = h // hpg
        cols += list(range(H * P + G * N + g * N, H * P + G * N + (g + 1) * N))
    cols = np.array(cols)
    hh = np.array(heads)
    bb = np.array(batches)
    xbc = f64(cpu["xbc"])[bb][:, :, cols]
    cs = f64(cpu.get("conv_state"))
    cs = cs[bb][:, :, cols] if (cs is not None and conv) else None
    z = f64(cpu.get("z"))
    if z is not None:
        zc = np.concatenate([np.arange(h * P, (h + 1) * P) for h in heads])
        z = z[bb][:, :, zc]
    h0 = f64(cpu.get("ssm_state"))
    h0 = h0[bb][:, hh] if h0 is not None else None
    nh = len(heads)
    y, hS, cs_out = oracle.mixer_prefill(
        xbc, f64(cpu["conv_w"])[cols] if conv else None, f64(cpu["dt_raw"])[bb][:, :, hh],
        f64(cpu["A"])[hh], H=nh, P=P, N=N, G=nh,
        conv_b=f64(cpu["conv_b"])[cols] if conv else None, conv_state=cs,
        dt_bias=f64(cpu["dt_bias"])[hh], D=f64(cpu["D"])[hh], z=z, h0=h0,
        dt_softplus=dt_softplus, nthreads=nthreads)
    return y, hS, cs_out, cols


class MaxRel:
    """max|gpu - oracle| / max|oracle| over a tensor compared piece by piece
    (the same number assert_close computes on the whole tensor), for outputs
    too large to hold in fp64 on the host at once."""

    def __init__(self, what):
        self.what, self.err, self.den, self.n = what, 0.0, 0.0, 0

    def add(self, gpu, ref):
        g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
        r = np.asarray(ref, np.float64)
        assert g.shape == r.shape, (self.what, g.shape, r.shape)
        assert np.all(np.isfinite(g)), f"{self.what}: non-finite GPU output"
        if g.size:
            self.err = max(self.err, float(np.max(np.abs(g - r))))
            self.den = max(self.den, float(np.max(np.abs(r))))
        self.n += g.size

    def check(self, tol, count):
        assert self.n == count, (self.what, self.n, count)
        e = self.err / self.den if self.den > 0 else self.err
        assert e <= tol, f"{self.what}: relative error {e:.3e} > {tol:.1e}"
        return e


def oracle_prefill_by_group(shape: si.Shape, cpu: dict, b: int, g: int, conv=True,
                            dt_softplus=True, nthreads=None):
    """fp64 oracle of sequence ``b`` for the heads of group ``g`` only, with the
    group's own B/C columns (one group per call keeps the fp64 copies of a
    long sequence small).  ``cpu`` holds host tensors [B, ...].  Returns
    (heads, y [S,hpg,P], hS [hpg,P,N], conv state [W-1, cols] or None, cols)."""
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    hpg = H // G
    heads = np.arange(g * hpg, (g + 1) * hpg)
    cols = np.concatenate([np.arange(g * hpg * P, (g + 1) * hpg * P),
                           H * P + g * N + np.arange(N),
                           H * P + G * N + g * N + np.arange(N)])
    tc, th = torch.from_numpy(cols), torch.from_numpy(heads)
    xbc = f64(cpu["xbc"][b][:, tc])[None]
    cs = cpu.get("conv_state")
    cs = f64(cs[b][:, tc])[None] if (cs is not None and conv) else None
    z = cpu.get("z")
    z = f64(z[b][:, g * hpg * P:(g + 1) * hpg * P])[None] if z is not None else None
    h0 = cpu.get("ssm_state")
    h0 = f64(h0[b][th])[None] if h0 is not None else None
    y, hS, cs_out = oracle.mixer_prefill(
        xbc, f64(cpu["conv_w"][tc]) if conv else None, f64(cpu["dt_raw"][b][:, th])[None],
        f64(cpu["A"][th]), H=hpg, P=P, N=N, G=1,
        conv_b=f64(cpu["conv_b"][tc]) if conv else None, conv_state=cs,
        dt_bias=f64(cpu["dt_bias"][th]), D=f64(cpu["D"][th]), z=z, h0=h0,
        dt_softplus=dt_softplus, nthreads=nthreads)
    return heads, y[0], hS[0], (cs_out[0] if cs_out is not None else None), cols


def check_prefill_every_element(shape: si.Shape, cpu: dict, y, h, cs, act, batches=None,
                                conv=True, gpu_batch_of=None):
    """Compare every element of y and of the final SSM state of the listed
    sequences (all by default) with the oracle, one (sequence, group) at a
    time, and the conv state bit for bit.  ``gpu_batch_of[i]`` is the index in
    the GPU tensors of the i-th listed sequence (default: the same index)."""
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    batches = list(range(shape.batch)) if batches is None else list(batches)
    ey, eh = MaxRel("y"), MaxRel("ssm_state")
    for i, b in enumerate(batches):
        gb = b if gpu_batch_of is None else gpu_batch_of[i]
        for g in range(G):
            heads, yo, ho, co, cols = oracle_prefill_by_group(shape, cpu, b, g, conv=conv)
            h0_, h1_ = int(heads[0]), int(heads[-1]) + 1
            ey.add(y[gb, :, h0_:h1_], yo)
            eh.add(h[gb, h0_:h1_], ho)
            if conv and cs is not None:
                gcs = f64(cs[gb][:, torch.from_numpy(cols).to(cs.device)])
                assert np.array_equal(gcs, co), "conv state must be the raw rows, bit for bit"
    tol = TOL[act]
    n = len(batches)
    return (ey.check(tol, n * shape.seqlen * H * P), eh.check(tol, n * H * P * N))


def oracle_sequence(shape: si.Shape, cpu: dict, b: int, conv=True, dt_softplus=True):
    """The oracle's y [S,H,P] and final SSM state [H,P,N] of sequence ``b``
    over all heads, computed one group of heads at a time."""
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    y = np.empty((shape.seqlen, H, P))
    hS = np.empty((H, P, N))
    for g in range(G):
        heads, yo, ho, _, _ = oracle_prefill_by_group(shape, cpu, b, g, conv=conv,
                                                      dt_softplus=dt_softplus)
        y[:, heads] = yo
        hS[heads] = ho
    return y, hS
