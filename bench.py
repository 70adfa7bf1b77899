"""Benchmark of the SSD mixer core on GB300: chunked prefill tokens/s per layer
and decode-step state GB/s, each against the HBM roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one ssd_chunk_scan call (conv + SiLU + chunked scan + z gate, with
carried conv/SSM state) over the Nemotron-H-8B-shaped prefill workload
(B=1 sequence, S=2048 rows, 128-row chunks, H=128, P=64, N=128, G=8, W=4, bf16
activations, fp32 state).  Inputs rotate over several resident sets whose
total exceeds the 129 MB L2, so no step reads its inputs from L2.  The decode
step (256 rows at slots of a 1024-slot fp32 pool [1024,128,64,128], conv pool
fused, 64 successive steps) is measured in the same run and reported under
"decode".  Under torchrun every rank runs its own replica (independent
sequences: weak scaling, no collective on the data path); the times are the
max over ranks.

--impl reference times the fp64 CPU oracle (the reference implementation of
this repository) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import ssd_inputs as si  # noqa: E402

METRIC = "SSD chunked-prefill tokens/s per layer; decode-step state GB/s vs HBM peak"
HBM_FALLBACK_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------------------
# algorithmic bytes (what one launch must move at minimum)

def prefill_bytes(shape: si.Shape, with_z=True) -> dict:
    """Per row: raw xBC + z + dt read, y written.  Per sequence: SSM state in
    and out (fp32) and conv state in and out."""
    e = 2  # bf16
    H, P, N, G, W = shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.conv_width
    per_row = shape.cdim * e + (H * P * e if with_z else 0) + H * 4 + H * P * e
    per_seq = 2 * H * P * N * 4 + 2 * (W - 1) * shape.cdim * e
    total = shape.batch * (shape.seqlen * per_row + per_seq)
    return {"per_row": per_row, "per_seq": per_seq, "per_launch": total}


def decode_state_bytes(rows, shape: si.Shape) -> int:
    return 2 * rows * shape.nheads * shape.headdim * shape.dstate * 4


def decode_other_bytes(rows, shape: si.Shape) -> int:
    e = 2
    H, P, C, W = shape.nheads, shape.headdim, shape.cdim, shape.conv_width
    return rows * (C * e + H * P * e + H * 4 + H * P * e + 2 * (W - 1) * C * e)


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return HBM_FALLBACK_GBS, "fallback"


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    cdir = os.path.join(ROOT, "ssd_scan_gb300", "csrc")
    for n in sorted(os.listdir(cdir)):
        if n.endswith((".cu", ".cuh")):
            with open(os.path.join(cdir, n), "rb") as f:
                h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kind: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            tr = json.load(f)
        ent = tr.get(kind)
        if ent and ent.get("source_sha") == kernel_source_sha():
            return ent.get("bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


# ---------------------------------------------------------------------------
# clocks sampled during the timed region

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.t:
                self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------

def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v: float, world: int, device="cuda") -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank: int) -> int:
    """Each rank draws its own independent sequences (weak scaling)."""
    return 1000 * rank


def whole_job_tokens_per_s(world: int, shape: si.Shape, ms_max: float) -> float:
    """Tokens all ranks processed in one step over the slowest rank's time."""
    return world * shape.batch * shape.seqlen / (ms_max / 1e3)


def queue_ahead(host_s_per_call: float, calls: int):
    """Keep the GPU busy (a spin kernel on the current stream) for longer than
    the host needs to queue `calls` calls, so that the start event recorded
    after it fires with the timed calls already queued: the events then time
    the device's work back to back, not the host's launch latency (the e2e
    number carries that)."""
    seconds = min(0.05, 2.0 * host_s_per_call * calls + 2e-4)
    torch.cuda._sleep(int(seconds * 2.1e9))  # cycles at up to 2.1 GHz


def make_prefill_sets(shape, nsets, seed_base, device):
    import ssd_scan_gb300 as ssd
    prm = {k: v.to(device) for k, v in si.params(shape, seed=seed_base).items()}
    sets = []
    d = ssd.dims(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                 shape.ngroups, shape.conv_width, shape.chunk)
    flags = ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z
    for i in range(nsets):
        inp = si.prefill_inputs(shape, seed=seed_base + 1 + i, device=device)
        B, S, H, P, N = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate
        out = {
            "y": torch.empty((B, S, H, P), dtype=torch.bfloat16, device=device),
            "hS": torch.empty((B, H, P, N), dtype=torch.float32, device=device),
            "cs": torch.empty((B, shape.conv_width - 1, shape.cdim), dtype=torch.bfloat16,
                              device=device),
        }
        ws = ssd.workspace_for(d, ssd.SSD_BF16, flags, True, device)
        sets.append((inp, out, ws))
    return prm, sets, d, flags


def prefill_call(ssd, d, flags, prm, inp, out, ws, stream):
    ssd.ssd_chunk_scan(d, ssd.SSD_BF16, flags, inp["xbc"], prm["conv_w"], prm["conv_b"],
                       inp["conv_state"], out["cs"], inp["dt_raw"], prm["dt_bias"], prm["A"],
                       prm["D"], inp["z"], inp["ssm_state"], out["y"], out["hS"], ws, stream)


def bench_ours(args):
    import ssd_scan_gb300 as ssd

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    ssd.load_library()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    if args.only == "decode":
        dec = bench_decode(ssd, dev, stream, world, args)
        return {"metric": "decode-step state GB/s", "decode": dec} if rank == 0 else None
    shape = si.PREFILL
    pb = prefill_bytes(shape)
    set_bytes = pb["per_launch"]
    nsets = max(3, -(-2 * L2_BYTES // set_bytes))  # rotate over > 2x L2 of inputs+outputs
    prm, sets, d, flags = make_prefill_sets(shape, nsets, rank_seed(rank), dev)

    # ---- warm-up (also the host's cost of one call), then K timed steps (one
    # ssd_chunk_scan call each), queued behind a spin so that none waits on the host
    host_s = []
    for i in range(args.warmup):
        inp, out, ws = sets[i % nsets]
        t0 = time.perf_counter()
        prefill_call(ssd, d, flags, prm, inp, out, ws, stream)
        host_s.append(time.perf_counter() - t0)
    torch.cuda.synchronize()
    host_call = statistics.median(host_s[1:] or host_s)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = ssd.ssd_launch_counts()
    with ClockSampler(local) as clk:
        _barrier(world)
        torch.cuda.synchronize()
        queue_ahead(host_call, args.steps)
        ev0.record(stream)
        t0 = time.perf_counter()
        for i in range(args.steps):
            inp, out, ws = sets[i % nsets]
            prefill_call(ssd, d, flags, prm, inp, out, ws, stream)
        host_loop = (time.perf_counter() - t0) / args.steps
        ev1.record(stream)
        torch.cuda.synchronize()
        _barrier(world)
    launches1 = ssd.ssd_launch_counts()
    ms = ev0.elapsed_time(ev1) / args.steps
    ms = _max_over_ranks(ms, world)
    gpu_launches = sum(launches1[k] - launches0[k] for k in launches0)
    value = whole_job_tokens_per_s(world, shape, ms)

    hbm, hbm_src = measured_peaks()
    achieved = pb["per_launch"] / (ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": ncu_traffic("prefill"),
                "peak_source": hbm_src,
                "kernel": "ssd_chunk_scan call (all its kernels, events around the call)",
                "algorithmic_bytes_per_launch": pb["per_launch"]}
    extra = None
    if args.only == "prefill":  # profiling runs: the timed prefill steps alone
        e2e = dec = None
    else:
        if args.extra:
            extra = bench_extra(ssd, dev, stream, args)
        # ---- end to end through the C-ABI from pinned host buffers
        e2e = bench_e2e(ssd, shape, d, flags, prm, sets[0], stream, args)
        # ---- decode step (256 rows, 1024-slot pool, 64 steps)
        dec = bench_decode(ssd, dev, stream, world, args)

    out = None
    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "nemotron-h-8b mixer prefill: B=1 x S=2048 rows per GPU, "
                                   "chunk 128, H=128 P=64 N=128 G=8 W=4, conv+SiLU and z-gate "
                                   "fused, carried conv/ssm state",
                       "batch_per_gpu": shape.batch, "seq_len": shape.seqlen,
                       "parallelism": f"replicas x{world} (independent sequences)",
                       "l2": f"inputs rotate over {nsets} resident sets "
                             f"({nsets * set_bytes / 1e6:.0f} MB > 129 MB L2)"},
            "roofline": roofline,
            "e2e": e2e,
            "gpu_launches": gpu_launches,
            "host_us_per_call": round(host_loop * 1e6, 1),
            "clocks": clk.summary(),
            "decode": dec,
        }
        if extra is not None:
            out["extra_workloads"] = extra
    return out


def bench_e2e(ssd, shape, d, flags, prm, dset, stream, args):
    """End to end through the C-ABI from pinned host buffers: every step copies
    its inputs host -> device, makes the ssd_chunk_scan call and copies its
    outputs device -> host, all inside the timed region.  The steps are
    pipelined the way a serving loop runs them: inputs go in on one copy
    stream, outputs come back on another, and the call runs on the compute
    stream, so step i+1's input copy and step i-1's output copy overlap step
    i's call (device inputs and outputs double-buffered, ordered by events).
    The same steps run one after the other are reported as `serial`."""
    inp, out, ws = dset
    host_in = {k: v.cpu().pin_memory() for k, v in inp.items() if v is not None}
    host_out = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out.items()}
                for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
    dev_in = [{k: torch.empty_like(v, device="cuda") for k, v in host_in.items()} for _ in range(2)]
    dev_out = [out, {k: torch.empty_like(v) for k, v in out.items()}]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    done, out_free = [ev(), ev()], [ev(), ev()]
    for e in in_free + out_free:
        e.record(stream)

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(in_free[b])  # the call of step i-2 is done with dev_in[b]
            for k, v in host_in.items():
                dev_in[b][k].copy_(v, non_blocking=True)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_free[b])  # step i-2's outputs have left dev_out[b]
        prefill_call(ssd, d, flags, prm, dev_in[b], dev_out[b], ws, stream)
        in_free[b].record(stream)
        done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b])
            for k, v in dev_out[b].items():
                host_out[b][k].copy_(v, non_blocking=True)
            out_free[b].record(s_out)

    def serial_step():
        for k, v in host_in.items():
            dev_in[0][k].copy_(v, non_blocking=True)
        prefill_call(ssd, d, flags, prm, dev_in[0], dev_out[0], ws, stream)
        for k, v in dev_out[0].items():
            host_out[0][k].copy_(v, non_blocking=True)

    n = max(3, min(args.steps, 20))
    timing = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    # serial: one stream, each step's copies and call in turn
    for _ in range(max(3, args.warmup)):
        serial_step()
    torch.cuda.synchronize()
    e0, e1 = timing()
    e0.record(stream)
    for _ in range(n):
        serial_step()
    e1.record(stream)
    torch.cuda.synchronize()
    serial_ms = e0.elapsed_time(e1) / n
    # pipelined: every stream waits on the start event; the end event follows the
    # last output copy, which follows every call and (by stream order) every copy
    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = timing()
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(n):
        step(i)
    stream.wait_event(out_free[(n - 1) % 2])
    stream.wait_event(out_free[n % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    tok = shape.batch * shape.seqlen
    return {"value": round(tok / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "pipelined": "input copy, call and output copy of consecutive steps overlap "
                         "(two copy streams, double-buffered device tensors)",
            "serial": {"value": round(tok / (serial_ms / 1e3), 1), "ms_per_step": round(serial_ms, 4)}}


def chained_calls(ssd, shape, prm, inp, splits, device):
    """Pre-sliced, contiguous per-call inputs and outputs for a sequence fed as
    consecutive ssd_chunk_scan calls (rows `splits`), each call continuing from
    the previous one's SSM and conv state.  Returns a function that issues the
    calls once."""
    B, H, P, N, G, W = (shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                        shape.conv_width)
    flags = ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z
    calls, r0 = [], 0
    hs = [torch.empty((B, H, P, N), dtype=torch.float32, device=device) for _ in range(2)]
    cs = [torch.empty((B, W - 1, shape.cdim), dtype=torch.bfloat16, device=device)
          for _ in range(2)]
    ws = ssd.workspace_for(ssd.dims(B, max(splits), H, P, N, G, W, shape.chunk), ssd.SSD_BF16,
                           flags, True, device)
    for i, L in enumerate(splits):
        d = ssd.dims(B, L, H, P, N, G, W, shape.chunk)
        c = {"d": d, "xbc": inp["xbc"][:, r0:r0 + L].contiguous(),
             "dt": inp["dt_raw"][:, r0:r0 + L].contiguous(),
             "z": inp["z"][:, r0:r0 + L].contiguous(),
             "y": torch.empty((B, L, H, P), dtype=torch.bfloat16, device=device),
             "h_in": inp["ssm_state"] if i == 0 else hs[(i - 1) % 2], "h_out": hs[i % 2],
             "cs_in": inp["conv_state"] if i == 0 else cs[(i - 1) % 2], "cs_out": cs[i % 2]}
        calls.append(c)
        r0 += L

    def run(stream):
        for c in calls:
            ssd.ssd_chunk_scan(c["d"], ssd.SSD_BF16, flags, c["xbc"], prm["conv_w"],
                               prm["conv_b"], c["cs_in"], c["cs_out"], c["dt"], prm["dt_bias"],
                               prm["A"], prm["D"], c["z"], c["h_in"], c["y"], c["h_out"], ws,
                               stream)
    return run, len(calls)


def bench_extra(ssd, dev, stream, args):
    """The other prefill workloads, timed like the headline one: long (8
    sequences x 8192 rows, then a chained second call of 8192 rows each) and
    decay stress (4 x 4096 rows with decays up to ~1e4 per row, fed as calls of
    U{1..128} rows), tokens/s over all calls of one pass; and the gated group
    RMSNorm at the prefill width, GB/s against the HBM peak."""
    out = {}
    for name, shape, splits, stress in (
            ("long_8x8192_plus_8192", si.LONG.with_(seqlen=2 * si.LONG.seqlen),
             [si.LONG.seqlen, si.LONG.seqlen], False),
            ("stress_4x4096_calls_1_to_128", si.STRESS, si.random_splits(si.STRESS.seqlen, 5),
             True)):
        prm = {k: v.to(dev) for k, v in si.params(shape, seed=11, stress=stress).items()}
        inp = si.prefill_inputs(shape, seed=12, device=dev, stress=stress)
        run, ncalls = chained_calls(ssd, shape, prm, inp, splits, dev)
        host_s = []
        for _ in range(3):
            t0 = time.perf_counter()
            run(stream)
            host_s.append(time.perf_counter() - t0)
        torch.cuda.synchronize()
        steps = 5
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        queue_ahead(min(host_s), steps)
        ev0.record(stream)
        for _ in range(steps):
            run(stream)
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / steps
        rows = shape.batch * shape.seqlen
        out[name] = {"tokens_per_s": round(rows / (ms / 1e3), 1), "ms_per_pass": round(ms, 4),
                     "calls_per_pass": ncalls, "rows_per_pass": rows,
                     "host_ms_per_pass": round(min(host_s) * 1e3, 3)}
        del inp, run
    # packed sequences with states at pool slots: 16 sequences of log-uniform
    # 1..2048 rows (seeded), at slots of a 64-slot pool, a quarter of them fresh
    sh = si.PREFILL
    gl = torch.Generator().manual_seed(33)
    lens = [int(v) for v in torch.exp(torch.rand(16, generator=gl) * np.log(2048.0)).round()]
    T = sum(lens)
    H, P, N, G, W = sh.nheads, sh.headdim, sh.dstate, sh.ngroups, sh.conv_width
    prm = {k: v.to(dev) for k, v in si.params(sh, seed=31).items()}
    inp = si.prefill_inputs(sh.with_(seqlen=T), seed=32, device=dev)
    rows = {k: inp[k][0].contiguous() for k in ("xbc", "dt_raw", "z")}
    del inp
    nslots = 64
    spool = torch.randn((nslots, H, P, N), device=dev) * 0.1
    cpool = torch.randn((nslots, W - 1, sh.cdim), device=dev).to(torch.bfloat16)
    slots = torch.randperm(nslots, generator=gl)[:16].to(torch.int32).to(dev)
    init = (torch.arange(16) % 4 != 0).to(torch.int32).to(dev)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
    y = torch.empty((T, H, P), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(T * 2 * G * N * 2, dtype=torch.uint8, device=dev)
    d = ssd.dims(16, T, H, P, N, G, W)
    flags = ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z

    def varlen_call():
        ssd.ssd_chunk_scan_varlen(d, ssd.SSD_BF16, flags, cu, slots, init, nslots, rows["xbc"],
                                  prm["conv_w"], prm["conv_b"], cpool, rows["dt_raw"],
                                  prm["dt_bias"], prm["A"], prm["D"], rows["z"], spool, y, ws,
                                  stream)
    for _ in range(3):
        varlen_call()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    queue_ahead(50e-6, 10)
    ev0.record(stream)
    for _ in range(10):
        varlen_call()
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / 10
    out["varlen_16_sequences_1_to_2048_rows_at_slots"] = {
        "tokens_per_s": round(T / (ms / 1e3), 1), "ms_per_call": round(ms, 4), "rows": T,
        "lengths": lens}
    del rows, spool, cpool, y, ws
    # the gated group RMSNorm after the scan, at the prefill width (2048 rows x
    # 8192 channels, 8 groups): HBM-bound, y and z read, out written once
    sh = si.PREFILL
    C = sh.nheads * sh.headdim
    g = torch.Generator(device=dev).manual_seed(21)
    sets = [(torch.randn((1, sh.seqlen, C), generator=g, device=dev).to(torch.bfloat16),
             torch.randn((1, sh.seqlen, C), generator=g, device=dev).to(torch.bfloat16),
             torch.empty((1, sh.seqlen, C), dtype=torch.bfloat16, device=dev)) for _ in range(3)]
    w = torch.rand((C,), generator=g, device=dev) + 0.5
    d = ssd.dims(1, sh.seqlen, sh.nheads, sh.headdim, sh.dstate, sh.ngroups)
    for i in range(6):
        y, z, o = sets[i % 3]
        ssd.ssd_gated_group_rmsnorm(d, ssd.SSD_BF16, y, z, w, 1e-5, o, stream)
    torch.cuda.synchronize()
    steps = 30
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    queue_ahead(30e-6, steps)
    ev0.record(stream)
    for i in range(steps):
        y, z, o = sets[i % 3]
        ssd.ssd_gated_group_rmsnorm(d, ssd.SSD_BF16, y, z, w, 1e-5, o, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    nbytes = 3 * sh.seqlen * C * 2 + C * 4
    hbm, _ = measured_peaks()
    out["gated_group_rmsnorm_2048x8192"] = {
        "us_per_call": round(ms * 1e3, 2), "bytes_per_call": nbytes,
        "gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
        "frac_of_hbm": round(nbytes / (ms / 1e3) / 1e9 / hbm, 4)}
    assert ssd.ssd_read_device_error(stream) == ssd.SSD_OK
    return out


def bench_decode(ssd, dev, stream, world, args):
    shape = si.DECODE
    R, nslots = si.DECODE_ROWS, max(si.DECODE_ROWS, args.decode_slots)
    prm = {k: v.to(dev) for k, v in si.params(shape).items()}
    pools = {k: v.to(dev) for k, v in si.decode_pools(shape, nslots, device=dev).items()}
    nin = 8
    ins = [{k: v.to(dev) for k, v in si.decode_inputs(shape, t, device=dev).items()}
           for t in range(nin)]
    y = torch.empty((R, shape.nheads, shape.headdim), dtype=torch.bfloat16, device=dev)
    d = ssd.dims(R, 1, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                 shape.conv_width)
    flags = ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z

    def step(t):
        inp = ins[t % nin]
        ssd.ssd_decode_step(d, ssd.SSD_BF16, flags, inp["xbc"], prm["conv_w"], prm["conv_b"],
                            pools["conv_pool"], inp["dt_raw"], prm["dt_bias"], prm["A"],
                            prm["D"], inp["z"], pools["slot_ids"], nslots, pools["ssm_pool"], y,
                            stream)

    host_s = []
    for t in range(max(3, args.warmup)):
        t0 = time.perf_counter()
        step(t)
        host_s.append(time.perf_counter() - t0)
    torch.cuda.synchronize()
    steps = si.DECODE_STEPS
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    queue_ahead(statistics.median(host_s[1:]), steps)
    ev0.record(stream)
    for t in range(steps):
        step(t)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = _max_over_ranks(ev0.elapsed_time(ev1) / steps, world)
    hbm, src = measured_peaks()
    sb = decode_state_bytes(R, shape)
    gbs = sb / (ms / 1e3) / 1e9
    total = (sb + decode_other_bytes(R, shape)) / (ms / 1e3) / 1e9
    assert ssd.ssd_read_device_error(stream) == ssd.SSD_OK
    return {"metric": "decode-step state GB/s", "value": round(gbs * world, 1), "unit": "GB/s",
            "per_gpu_gbs": round(gbs, 1), "ms_per_step": round(ms, 5), "steps": steps,
            "rows": R, "slots": nslots, "state_bytes_per_step": sb,
            "all_bytes_gbs": round(total, 1), "peak": hbm, "peak_source": src,
            "frac": round(gbs / hbm, 4), "traffic": ncu_traffic("decode")}


# ---------------------------------------------------------------------------
# the fp64 oracle on the host cores

def oracle_sample_rows() -> int:
    return int(os.environ.get("SSD_BENCH_ORACLE_ROWS", str(si.PREFILL.seqlen)))


def oracle_prefill_sample(rows: int):
    """Time the oracle on the first ``rows`` rows of the prefill workload (all
    heads: conv + SiLU + recurrence + gate).  Returns (seconds, threads)."""
    import oracle
    import numpy as np
    shape = si.PREFILL.with_(seqlen=rows)
    prm = si.params(shape, seed=0)
    inp = si.prefill_inputs(shape, seed=1)
    f = lambda t: None if t is None else t.to(torch.float64).numpy()  # noqa: E731
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    args = (f(inp["xbc"]), f(prm["conv_w"]), f(inp["dt_raw"]), f(prm["A"]))
    kw = dict(H=H, P=P, N=N, G=G, conv_b=f(prm["conv_b"]), conv_state=f(inp["conv_state"]),
              dt_bias=f(prm["dt_bias"]), D=f(prm["D"]), z=f(inp["z"]), h0=f(inp["ssm_state"]))
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    y, h, c = oracle.mixer_prefill(*args, nthreads=threads, **kw)
    dt = time.perf_counter() - t0
    assert np.isfinite(y).all()
    return dt, threads


def cpu_baseline(min_seconds: float = 10.0) -> dict:
    """The oracle on the prefill workload, repeated until at least
    `min_seconds` of wall time (at least once)."""
    rows = oracle_sample_rows()
    total, passes, threads = 0.0, 0, 1
    while passes == 0 or total < min_seconds:
        dt, threads = oracle_prefill_sample(rows)
        total += dt
        passes += 1
    return {"value": round(rows * passes / total, 2), "unit": "tokens/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{passes} passes over the first {rows} of the 2048 rows of the prefill "
                      f"workload, all 128 heads (conv + recurrence + gate, fp64), {total:.1f} s"}


def bench_reference(args):
    rank, world, local = _dist()
    if rank != 0:
        return None
    rows = oracle_sample_rows()
    for _ in range(args.warmup):
        oracle_prefill_sample(rows)
    times = []
    threads = 1
    for _ in range(args.steps):
        dt, threads = oracle_prefill_sample(rows)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = rows / (ms / 1e3)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "nemotron-h-8b mixer prefill (as the main arm); each step is a "
                               f"bounded sample: the first {rows} rows, all 128 heads",
                   "batch_per_gpu": 1, "seq_len": rows, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": f"first {rows} rows x 128 heads per step"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra", action="store_true",
                    help="also time the long (8 x 8192 + 8192) and decay-stress prefill workloads")
    ap.add_argument("--only", choices=["all", "prefill", "decode"], default="all",
                    help="time only the prefill or only the decode steps (profiler runs)")
    ap.add_argument("--decode-slots", type=int, default=si.DECODE_SLOTS,
                    help="slots in the decode pool (the 256 rows touch the same bytes "
                         "whatever the pool size; a smaller pool keeps profiler captures small)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        res = bench_reference(args)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    res = bench_ours(args)
    rank, world, _ = _dist()
    if rank == 0 and res is not None:
        if world == 1 and not args.no_cpu_baseline and args.only == "all":
            res["cpu_baseline"] = cpu_baseline()
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
