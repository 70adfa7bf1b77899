"""Seeded synthetic inputs for the SSD mixer core (shared by tests and bench).

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and distributions of the workloads below.  Both the fp64
oracle (``oracle/``) and the CUDA library (``ssd_scan_gb300``) consume what it
produces; neither is imported here.

Distributions (the pages give no input data; this is the stated recipe):

* raw xBC rows (x | B | C stream before the conv) ~ N(0, 1)
* z ~ N(0, 1)
* dt_raw ~ N(0, 1); dt_bias chosen so that softplus(dt_bias) is log-uniform
  in [1e-3, 1e-1] (the inverse softplus below only places the draw)
* A = -exp(U(0, ln 16)), D ~ N(0, 1)
* conv weight ~ N(0, 1/W) (std W**-0.5), conv bias ~ N(0, 0.1**2)
* initial SSM state ~ N(0, 0.1**2) (fp32), initial conv state ~ N(0, 1)
* decay stress: dt_raw ~ N(4, 2**2), A = -exp(U(ln 1e3, ln 1e4))

Workloads (Nemotron-H-8B mixer shape: H=128 heads, P=64, N=128, G=8, W=4,
conv dim 8192 + 2*8*128 = 10240):

* ``tiny``      B=1, S=11, H=4, P=16, N=16, G=1, fp32, zero initial states
* ``prefill``   B=1, S=2048, bf16 activations, nonzero initial states
* ``long``      B=8, S=8192 (plus a second 8192-row call on the final states)
* ``stress``    B=4, S=4096, decay stress, rows split into 1..128-row calls
* ``decode``    256 rows in a 1024-slot pool, 64 steps
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Shape:
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    conv_width: int = 4
    chunk: int = 128

    @property
    def cdim(self) -> int:
        return self.nheads * self.headdim + 2 * self.ngroups * self.dstate

    def with_(self, **kw) -> "Shape":
        return dataclasses.replace(self, **kw)


NEMOTRON_H_8B = dict(nheads=128, headdim=64, dstate=128, ngroups=8, conv_width=4)

TINY = Shape(batch=1, seqlen=11, nheads=4, headdim=16, dstate=16, ngroups=1)
PREFILL = Shape(batch=1, seqlen=2048, **NEMOTRON_H_8B)
LONG = Shape(batch=8, seqlen=8192, **NEMOTRON_H_8B)
STRESS = Shape(batch=4, seqlen=4096, **NEMOTRON_H_8B)
DECODE_ROWS = 256
DECODE_SLOTS = 1024
DECODE_STEPS = 64
DECODE = Shape(batch=DECODE_ROWS, seqlen=1, **NEMOTRON_H_8B)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, g, device, mean=0.0, std=1.0):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(mean, std, generator=g)
    return t


def _uniform(shape, g, device, lo, hi):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.uniform_(lo, hi, generator=g)
    return t


def _dt_bias(nheads, g, device):
    # target v = softplus(bias) log-uniform in [1e-3, 1e-1]; bias = log(expm1(v))
    v = torch.exp(_uniform((nheads,), g, device, math.log(1e-3), math.log(1e-1)))
    return torch.log(torch.expm1(v.double())).float()


def params(shape: Shape, seed: int = 0, device="cpu", stress: bool = False) -> dict:
    """Per-layer parameters: conv_w [Cdim,W], conv_b [Cdim], dt_bias, A, D [H]."""
    g = _gen(seed + 7919, device)
    H, C, W = shape.nheads, shape.cdim, shape.conv_width
    out = {
        "conv_w": _normal((C, W), g, device, std=W ** -0.5),
        "conv_b": _normal((C,), g, device, std=0.1),
        "dt_bias": _dt_bias(H, g, device),
        "D": _normal((H,), g, device),
    }
    if stress:
        out["A"] = -torch.exp(_uniform((H,), g, device, math.log(1e3), math.log(1e4)))
    else:
        out["A"] = -torch.exp(_uniform((H,), g, device, 0.0, math.log(16.0)))
    return out


def prefill_inputs(shape: Shape, seed: int = 0, device="cpu", act_dtype=torch.bfloat16,
                   stress: bool = False, initial_state: bool = True,
                   with_z: bool = True) -> dict:
    """Activations of one prefill call: xbc raw [B,S,Cdim], z [B,S,H*P],
    dt_raw [B,S,H], ssm_state [B,H,P,N] fp32 (or None), conv_state
    [B,W-1,Cdim] (or None)."""
    g = _gen(seed, device)
    B, S, H, P, N = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate
    C, W = shape.cdim, shape.conv_width
    out = {"xbc": _normal((B, S, C), g, device).to(act_dtype)}
    out["z"] = _normal((B, S, H * P), g, device).to(act_dtype) if with_z else None
    if stress:
        out["dt_raw"] = _normal((B, S, H), g, device, mean=4.0, std=2.0)
    else:
        out["dt_raw"] = _normal((B, S, H), g, device)
    if initial_state:
        out["ssm_state"] = _normal((B, H, P, N), g, device, std=0.1)
        out["conv_state"] = _normal((B, W - 1, C), g, device).to(act_dtype)
    else:
        out["ssm_state"] = None
        out["conv_state"] = None
    return out


def decode_pools(shape: Shape, num_slots: int, seed: int = 0, device="cpu",
                 act_dtype=torch.bfloat16) -> dict:
    """Slot pools: ssm_pool [num_slots,H,P,N] fp32 ~ N(0, 0.1^2), conv_pool
    [num_slots,W-1,Cdim] ~ N(0,1), and slot_ids = the first ``batch`` entries
    of a seeded permutation of the slots (int32)."""
    g = _gen(seed + 104729, device)
    H, P, N, C, W = shape.nheads, shape.headdim, shape.dstate, shape.cdim, shape.conv_width
    ssm_pool = _normal((num_slots, H, P, N), g, device, std=0.1)
    conv_pool = _normal((num_slots, W - 1, C), g, device).to(act_dtype)
    gc = _gen(seed, "cpu")
    perm = torch.randperm(num_slots, generator=gc)[: shape.batch].to(torch.int32)
    return {"ssm_pool": ssm_pool, "conv_pool": conv_pool, "slot_ids": perm.to(device)}


def decode_inputs(shape: Shape, step: int, seed: int = 0, device="cpu",
                  act_dtype=torch.bfloat16, with_z: bool = True) -> dict:
    """Activations of decode step ``step``: xbc raw [R,Cdim], z [R,H*P],
    dt_raw [R,H]."""
    g = _gen(seed * 1000003 + 31 * step + 1, device)
    R, H, P, C = shape.batch, shape.nheads, shape.headdim, shape.cdim
    return {
        "xbc": _normal((R, C), g, device).to(act_dtype),
        "z": _normal((R, H * P), g, device).to(act_dtype) if with_z else None,
        "dt_raw": _normal((R, H), g, device),
    }


def random_splits(total: int, seed: int, lo: int = 1, hi: int = 128) -> list[int]:
    """A seeded split of ``total`` rows into calls of U{lo..hi} rows."""
    g = torch.Generator()
    g.manual_seed(int(seed) + 15485863)
    out, left = [], total
    while left > 0:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g))
        n = min(n, left)
        out.append(n)
        left -= n
    return out
