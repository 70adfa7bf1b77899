"""Benchmark of the SSD mixer core on GB300: chunked prefill tokens/s per layer
and decode-step state GB/s, each against the HBM roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the long-prefill workload: 8 independent sequences x
8192 rows in one ssd_chunk_scan call (conv + SiLU + chunked scan + z gate,
carried conv/SSM state), then a second 8192-row call of each sequence fed
with the first call's final states (Nemotron-H-8B mixer: 128-row chunks,
H=128, P=64, N=128, G=8, W=4, bf16 activations, fp32 state).  Its inputs
(7 GB) are far larger than the 129 MB L2.  The same run also reports the
2048-row single-sequence prefill (inputs rotating over resident sets larger
than L2) under "prefill_2048", and the decode step (256 rows at slots of a
1024-slot fp32 pool [1024,128,64,128], conv pool fused, 64 successive steps)
under "decode".  Under torchrun every rank runs its own replica (independent
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
    """Hash of the kernel sources and of the build script (its flags shape the
    code as well)."""
    h = hashlib.sha256()
    cdir = os.path.join(ROOT, "ssd_scan_gb300", "csrc")
    for n in sorted(os.listdir(cdir)):
        if n.endswith((".cu", ".cuh")):
            with open(os.path.join(cdir, n), "rb") as f:
                h.update(n.encode() + f.read())
    with open(os.path.join(ROOT, "ssd_scan_gb300", "build.py"), "rb") as f:
        h.update(b"build.py" + f.read())
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
        self.lines = []  # (host time, line)
        self.t = None
        self.window = None  # (t0, t1) of the timed region, host clock

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, t0: float, t1: float):
        """The timed region, on the host clock: only samples read inside it
        (with 50 ms of slack for the sampler's own latency) are summarised,
        when there are any."""
        self.window = (t0 - 0.05, t1 + 0.05)

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
        lines = [ln for t, ln in self.lines]
        if self.window is not None:
            inside = [ln for t, ln in self.lines if self.window[0] <= t <= self.window[1]]
            lines = inside or lines
        for ln in lines:
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


LONG_STEP = si.LONG.with_(seqlen=2 * si.LONG.seqlen)  # two chained calls of 8192 rows
LONG_SPLITS = [si.LONG.seqlen, si.LONG.seqlen]


def long_step_bytes(batch: int = si.LONG.batch) -> dict:
    """Algorithmic bytes of one long step: two calls of batch x 8192 rows,
    each with its per-row bytes and its per-sequence state bytes."""
    pb = prefill_bytes(si.LONG.with_(batch=batch))
    per_call = pb["per_launch"]
    return {"per_row": pb["per_row"], "per_seq_per_call": pb["per_seq"], "per_call": per_call,
            "per_step": len(LONG_SPLITS) * per_call}


def bench_long(ssd, dev, stream, world, rank, args):
    """The headline: K steps of the long workload (two chained calls each),
    queued behind a spin so that none waits on the host, timed with CUDA
    events on the launching stream; clocks sampled during the timed loop."""
    shape = LONG_STEP.with_(batch=args.long_batch)
    prm = {k: v.to(dev) for k, v in si.params(shape, seed=rank_seed(rank)).items()}
    inp = si.prefill_inputs(shape, seed=rank_seed(rank) + 1, device=dev)
    run, ncalls = chained_calls(ssd, shape, prm, inp, LONG_SPLITS, dev)
    host_s = []
    for _ in range(args.warmup):
        t0 = time.perf_counter()
        run(stream)
        host_s.append(time.perf_counter() - t0)
    torch.cuda.synchronize()
    host_step = statistics.median(host_s[1:] or host_s)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = ssd.ssd_launch_counts()
    with ClockSampler(torch.cuda.current_device()) as clk:
        _barrier(world)
        torch.cuda.synchronize()
        queue_ahead(host_step, args.steps)
        ev0.record(stream)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            run(stream)
        host_loop = (time.perf_counter() - t0) / args.steps
        ev1.record(stream)
        torch.cuda.synchronize()
        clk.mark(t0, time.perf_counter())
        _barrier(world)
    launches1 = ssd.ssd_launch_counts()
    assert ssd.ssd_read_device_error(stream) == ssd.SSD_OK
    ms = _max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
    nb = long_step_bytes(args.long_batch)
    hbm, hbm_src = measured_peaks()
    achieved = nb["per_step"] / (ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": ncu_traffic("long"),
                "peak_source": hbm_src,
                "kernel": "one ssd_chunk_scan call of 8 x 8192 rows (its B|C conv and scan "
                          "kernels; events around the calls, two equal calls per step)",
                "algorithmic_bytes_per_launch": nb["per_call"],
                "algorithmic_bytes_per_row": nb["per_row"],
                "algorithmic_state_bytes_per_sequence": nb["per_seq_per_call"],
                "ms_per_launch": round(ms / ncalls, 5)}
    del run, inp
    return {"ms": ms, "value": whole_job_tokens_per_s(world, shape, ms), "roofline": roofline,
            "gpu_launches": sum(launches1[k] - launches0[k] for k in launches0),
            "host_us_per_step": round(host_loop * 1e6, 1), "clocks": clk.summary()}


def bench_prefill_2048(ssd, dev, stream, world, rank, args):
    """The 2048-row single-sequence prefill, one ssd_chunk_scan call per step,
    inputs rotating over resident sets whose total exceeds twice the L2."""
    shape = si.PREFILL
    pb = prefill_bytes(shape)
    set_bytes = pb["per_launch"]
    nsets = max(3, -(-2 * L2_BYTES // set_bytes))
    prm, sets, d, flags = make_prefill_sets(shape, nsets, rank_seed(rank), dev)
    host_s = []
    for i in range(args.warmup):
        inp, out, ws = sets[i % nsets]
        t0 = time.perf_counter()
        prefill_call(ssd, d, flags, prm, inp, out, ws, stream)
        host_s.append(time.perf_counter() - t0)
    torch.cuda.synchronize()
    host_call = statistics.median(host_s[1:] or host_s)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    queue_ahead(host_call, args.steps)
    ev0.record(stream)
    for i in range(args.steps):
        inp, out, ws = sets[i % nsets]
        prefill_call(ssd, d, flags, prm, inp, out, ws, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = _max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
    hbm, hbm_src = measured_peaks()
    achieved = pb["per_launch"] / (ms / 1e3) / 1e9
    res = {"workload": "B=1 x S=2048 rows, one ssd_chunk_scan call per step",
           "tokens_per_s": round(whole_job_tokens_per_s(world, shape, ms), 1),
           "ms_per_call": round(ms, 5),
           "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                        "unit": "GB/s", "frac": round(achieved / hbm, 4),
                        "traffic": ncu_traffic("prefill"), "peak_source": hbm_src,
                        "algorithmic_bytes_per_launch": pb["per_launch"]},
           "l2": f"inputs rotate over {nsets} resident sets "
                 f"({nsets * set_bytes / 1e6:.0f} MB > 129 MB L2)"}
    return res, (shape, d, flags, prm, sets[0])


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
    if args.only == "tail":  # profiling runs: the scan + gated norm calls alone
        tail = {"mixer_tail_2048": bench_mixer_tail(ssd, dev, stream, si.PREFILL, steps=args.steps)}
        return {"metric": "mixer_tail", **tail} if rank == 0 else None
    if args.only == "stress":  # profiling runs: the decay-stress passes alone
        st = {"stress_4x4096_calls_1_to_128": bench_stress(ssd, dev, stream, steps=args.steps)}
        return {"metric": "stress", **st} if rank == 0 else None
    if args.only == "prefill":  # profiling runs: the 2048-row calls alone
        p2048, _ = bench_prefill_2048(ssd, dev, stream, world, rank, args)
        return {"metric": "prefill_2048", "prefill_2048": p2048} if rank == 0 else None
    head = bench_long(ssd, dev, stream, world, rank, args)
    extra = e2e = dec = p2048 = None
    if args.only == "all":
        p2048, _ = bench_prefill_2048(ssd, dev, stream, world, rank, args)
        if not args.no_extra:
            extra = bench_extra(ssd, dev, stream, args)
        # ---- end to end through the C-ABI from pinned host buffers
        e2e = bench_e2e_long(ssd, dev, stream, rank, args)
        # ---- decode step (256 rows, 1024-slot pool, 64 steps)
        dec = bench_decode(ssd, dev, stream, world, args)

    out = None
    if rank == 0:
        shape = LONG_STEP
        out = {
            "metric": METRIC, "value": round(head["value"], 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(head["ms"], 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "nemotron-h-8b mixer long prefill: 8 sequences x 8192 rows "
                                   "per GPU in one call, then a second 8192-row call of each fed "
                                   "with the final conv/ssm states; chunk 128, H=128 P=64 N=128 "
                                   "G=8 W=4, conv+SiLU and z-gate fused",
                       "batch_per_gpu": args.long_batch, "seq_len": shape.seqlen,
                       "calls_per_step": len(LONG_SPLITS),
                       "parallelism": f"replicas x{world} (independent sequences)",
                       "l2": "inputs of one step 7.2 GB > 129 MB L2"},
            "roofline": head["roofline"],
            "e2e": e2e,
            "gpu_launches": head["gpu_launches"],
            "host_us_per_step": head["host_us_per_step"],
            "clocks": head["clocks"],
            "prefill_2048": p2048,
            "decode": dec,
        }
        if extra is not None:
            out["extra_workloads"] = extra
    return out


def link_rates(dev, nbytes: int = 1 << 30) -> dict:
    """The host link's copy rates on this machine, from pinned host memory by the
    copy engines: host -> device alone, device -> host alone, and both at once
    (GB/s per direction), each the best of three 1 GiB copies."""
    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def best_ms(h2d: bool, d2h: bool) -> float:
        best = float("inf")
        for _ in range(3):
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            torch.cuda.synchronize()
            e0.record(s1)
            s2.wait_event(e0)
            if h2d:
                with torch.cuda.stream(s1):
                    d_a.copy_(h_in, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s2):
                    h_out.copy_(d_b, non_blocking=True)
            e2.record(s2)
            s1.wait_event(e2)
            e1.record(s1)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return best

    gbs = lambda ms: round(nbytes / (ms / 1e3) / 1e9, 1)  # noqa: E731
    out = {"h2d_gbs": gbs(best_ms(True, False)), "d2h_gbs": gbs(best_ms(False, True)),
           "both_ways_gbs_per_direction": gbs(best_ms(True, True))}
    del h_in, h_out, d_a, d_b
    torch.cuda.empty_cache()
    return out


def link_bound_ms(h2d_bytes: int, d2h_bytes: int, link: dict) -> float:
    """Least time per step the link allows: the shorter direction's bytes at
    the both-ways rate, with as many bytes of the longer one beside them, and
    the rest of the longer direction at its own rate."""
    both = link["both_ways_gbs_per_direction"] * 1e9
    lo = min(h2d_bytes, d2h_bytes)
    rest = max(h2d_bytes, d2h_bytes) - lo
    alone = (link["h2d_gbs"] if h2d_bytes >= d2h_bytes else link["d2h_gbs"]) * 1e9
    return (lo / both + rest / alone) * 1e3


def bench_e2e_long(ssd, dev, stream, rank, args):
    """End to end through the C-ABI from pinned host buffers: every step copies
    its inputs (the rows of both calls and the initial states) host -> device,
    makes the two chained ssd_chunk_scan calls and copies y and the final
    states device -> host, all inside the timed region.  Steps are pipelined
    as a serving loop runs them: inputs go in on one copy stream, outputs come
    back on another, the calls run on the compute stream, device tensors are
    double-buffered and ordered by events, so one step's copies overlap the
    neighbouring steps' calls.  The same steps run one after the other are
    reported as `serial`."""
    shape = LONG_STEP
    B, H, P, N, G, W = (shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                        shape.conv_width)
    L = si.LONG.seqlen
    prm = {k: v.to(dev) for k, v in si.params(shape, seed=rank_seed(rank)).items()}
    src = si.prefill_inputs(shape, seed=rank_seed(rank) + 1, device=dev)
    rows = ("xbc", "dt_raw", "z")
    # host inputs per call (each call's rows contiguous, so every copy is one
    # contiguous pinned transfer) and the initial states
    host_in = {"calls": [{k: src[k][:, c * L:(c + 1) * L].contiguous().cpu().pin_memory()
                          for k in rows} for c in range(2)],
               "ssm_state": src["ssm_state"].cpu().pin_memory(),
               "conv_state": src["conv_state"].cpu().pin_memory()}
    del src
    flags = ssd.SSD_DT_SOFTPLUS | ssd.SSD_HAS_Z
    d = ssd.dims(B, L, H, P, N, G, W, shape.chunk)
    ws = ssd.workspace_for(d, ssd.SSD_BF16, flags, True, dev)

    def dev_set():
        ins = {"calls": [{k: torch.empty_like(v, device=dev) for k, v in hc.items()}
                         for hc in host_in["calls"]],
               "ssm_state": torch.empty_like(host_in["ssm_state"], device=dev),
               "conv_state": torch.empty_like(host_in["conv_state"], device=dev)}
        outs = {"y": [torch.empty((B, L, H, P), dtype=torch.bfloat16, device=dev)
                      for _ in range(2)],
                "hS": [torch.empty((B, H, P, N), dtype=torch.float32, device=dev)
                       for _ in range(2)],
                "cs": [torch.empty((B, W - 1, shape.cdim), dtype=torch.bfloat16, device=dev)
                       for _ in range(2)]}
        return ins, outs

    sets = [dev_set(), dev_set()]
    host_out = [{"y": [torch.empty((B, L, H, P), dtype=torch.bfloat16, pin_memory=True)
                       for _ in range(2)],
                 "hS": torch.empty((B, H, P, N), dtype=torch.float32, pin_memory=True),
                 "cs": torch.empty((B, W - 1, shape.cdim), dtype=torch.bfloat16,
                                   pin_memory=True)} for _ in range(2)]
    nbytes = lambda t: t.numel() * t.element_size()  # noqa: E731
    h2d = sum(nbytes(v) for hc in host_in["calls"] for v in hc.values()) + \
        nbytes(host_in["ssm_state"]) + nbytes(host_in["conv_state"])
    d2h = sum(nbytes(v) for v in host_out[0]["y"]) + nbytes(host_out[0]["hS"]) + \
        nbytes(host_out[0]["cs"])

    def copy_in(ins):
        ins["ssm_state"].copy_(host_in["ssm_state"], non_blocking=True)
        ins["conv_state"].copy_(host_in["conv_state"], non_blocking=True)
        for c in range(2):
            for k in rows:
                ins["calls"][c][k].copy_(host_in["calls"][c][k], non_blocking=True)

    def calls(ins, outs, st):
        for c in range(2):
            ci = ins["calls"][c]
            ssd.ssd_chunk_scan(d, ssd.SSD_BF16, flags, ci["xbc"], prm["conv_w"], prm["conv_b"],
                               ins["conv_state"] if c == 0 else outs["cs"][0], outs["cs"][c],
                               ci["dt_raw"], prm["dt_bias"], prm["A"], prm["D"], ci["z"],
                               ins["ssm_state"] if c == 0 else outs["hS"][0], outs["y"][c],
                               outs["hS"][c], ws, st)

    def copy_out(outs, ho):
        for c in range(2):
            ho["y"][c].copy_(outs["y"][c], non_blocking=True)
        ho["hS"].copy_(outs["hS"][1], non_blocking=True)
        ho["cs"].copy_(outs["cs"][1], non_blocking=True)

    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    done, out_free = [ev(), ev()], [ev(), ev()]
    for e in in_free + out_free:
        e.record(stream)

    def step(i):
        b = i % 2
        ins, outs = sets[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(in_free[b])
            copy_in(ins)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_free[b])
        calls(ins, outs, stream)
        in_free[b].record(stream)
        done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b])
            copy_out(outs, host_out[b])
            out_free[b].record(s_out)

    def serial_step():
        ins, outs = sets[0]
        copy_in(ins)
        calls(ins, outs, stream)
        copy_out(outs, host_out[0])

    n = max(10, min(args.steps, 50))  # pipeline fill and drain amortised over >= 10 steps
    timing = lambda: (torch.cuda.Event(enable_timing=True),  # noqa: E731
                      torch.cuda.Event(enable_timing=True))
    for _ in range(3):
        serial_step()
    torch.cuda.synchronize()
    e0, e1 = timing()
    e0.record(stream)
    for _ in range(n):
        serial_step()
    e1.record(stream)
    torch.cuda.synchronize()
    serial_ms = e0.elapsed_time(e1) / n
    for i in range(3):
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
    assert ssd.ssd_read_device_error(stream) == ssd.SSD_OK
    tok = shape.batch * shape.seqlen
    del sets, host_out, host_in
    torch.cuda.empty_cache()
    link = link_rates(dev)
    bound = link_bound_ms(h2d, d2h, link)
    link["step_ms_bound"] = round(bound, 3)
    link["frac_of_bound"] = round(bound / ms, 4)
    return {"value": round(tok / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "steps": n,
            "pipelined": "input copy, calls and output copy of consecutive steps overlap "
                         "(two copy streams, double-buffered device tensors)",
            "serial": {"value": round(tok / (serial_ms / 1e3), 1),
                       "ms_per_step": round(serial_ms, 4)},
            "link": link}


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


def bench_stress(ssd, dev, stream, steps):
    """The decay-stress workload: 4 x 4096 rows with decays up to ~1e4 per
    row, fed as chained calls of U{1..128} rows (seeded splits); tokens/s
    over all calls of one pass."""
    shape, splits = si.STRESS, si.random_splits(si.STRESS.seqlen, 5)
    prm = {k: v.to(dev) for k, v in si.params(shape, seed=11, stress=True).items()}
    inp = si.prefill_inputs(shape, seed=12, device=dev, stress=True)
    run, ncalls = chained_calls(ssd, shape, prm, inp, splits, dev)
    host_s = []
    for _ in range(3):
        t0 = time.perf_counter()
        run(stream)
        host_s.append(time.perf_counter() - t0)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    queue_ahead(min(host_s), steps)
    ev0.record(stream)
    for _ in range(steps):
        run(stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    rows = shape.batch * shape.seqlen
    return {"tokens_per_s": round(rows / (ms / 1e3), 1), "ms_per_pass": round(ms, 4),
            "calls_per_pass": ncalls, "rows_per_pass": rows,
            "host_ms_per_pass": round(min(host_s) * 1e3, 3)}


def bench_extra(ssd, dev, stream, args):
    """The other workloads, timed like the headline one: decay stress (4 x
    4096 rows with decays up to ~1e4 per row, fed as calls of U{1..128} rows),
    tokens/s over all calls of one pass; 16 packed sequences at pool slots
    (one ssd_chunk_scan_varlen call); and the gated group RMSNorm at the
    prefill width, GB/s against the HBM peak."""
    out = {"stress_4x4096_calls_1_to_128": bench_stress(ssd, dev, stream, steps=5)}
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
    out["mixer_tail_2048"] = bench_mixer_tail(ssd, dev, stream, si.PREFILL, steps=30)
    out["mixer_tail_8x8192"] = bench_mixer_tail(ssd, dev, stream, si.LONG, steps=6)
    assert ssd.ssd_read_device_error(stream) == ssd.SSD_OK
    return out


def bench_mixer_tail(ssd, dev, stream, shape, steps):
    """The scan with the gated group RMSNorm after it: one
    ssd_chunk_scan_gated_norm call (the gate and the per-head sums of squares
    in the scan's epilogue, a scale pass after it) against ssd_chunk_scan
    without the gate followed by ssd_gated_group_rmsnorm in place, on the
    same inputs rotating over resident sets larger than the L2."""
    pb = prefill_bytes(shape)
    nsets = max(3, -(-2 * L2_BYTES // pb["per_launch"]))
    prm, sets, d, _ = make_prefill_sets(shape, nsets, 41, dev)
    H, C, S = shape.nheads, shape.nheads * shape.headdim, shape.batch * shape.seqlen
    w = torch.rand((C,), generator=torch.Generator(device=dev).manual_seed(42), device=dev) + 0.5
    fl = ssd.SSD_DT_SOFTPLUS
    wsn = [ssd.workspace_for(d, ssd.SSD_BF16, fl | ssd.SSD_GATED_NORM, True, dev) for _ in sets]

    def fused(i):
        inp, out, _ = sets[i % nsets]
        ssd.ssd_chunk_scan_gated_norm(
            d, ssd.SSD_BF16, fl, inp["xbc"], prm["conv_w"], prm["conv_b"], inp["conv_state"],
            out["cs"], inp["dt_raw"], prm["dt_bias"], prm["A"], prm["D"], inp["z"], w, 1e-5,
            inp["ssm_state"], out["y"], out["hS"], wsn[i % nsets], stream)

    def unfused(i):
        inp, out, ws = sets[i % nsets]
        ssd.ssd_chunk_scan(d, ssd.SSD_BF16, fl, inp["xbc"], prm["conv_w"], prm["conv_b"],
                           inp["conv_state"], out["cs"], inp["dt_raw"], prm["dt_bias"], prm["A"],
                           prm["D"], None, inp["ssm_state"], out["y"], out["hS"], ws, stream)
        ssd.ssd_gated_group_rmsnorm(d, ssd.SSD_BF16, out["y"], inp["z"], w, 1e-5, out["y"],
                                    stream)

    def timed(fn):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        queue_ahead(60e-6, steps)
        ev0.record(stream)
        for i in range(steps):
            fn(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / steps

    ms_f, ms_u = timed(fused), timed(unfused)
    # the fused call moves the scan's bytes, y once more in and out (the scale
    # pass) and the per-head sums of squares out and in
    nbytes = pb["per_launch"] + 2 * S * C * 2 + 2 * S * H * 4
    hbm, _ = measured_peaks()
    del sets, wsn
    return {"workload": f"B={shape.batch} x S={shape.seqlen} rows, one call per step",
            "fused_us_per_call": round(ms_f * 1e3, 2),
            "scan_then_norm_us_per_call": round(ms_u * 1e3, 2),
            "speedup": round(ms_u / ms_f, 3),
            "fused_tokens_per_s": round(S / (ms_f / 1e3), 1),
            "fused_algorithmic_bytes": nbytes,
            "fused_frac_of_hbm": round(nbytes / (ms_f / 1e3) / 1e9 / hbm, 4)}


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
    # K tokens of every row in one call (multi-token decode): the state moves
    # once per call, so tokens/s grows with K while the call stays HBM-bound
    multi = {}
    for K in (2, 4, 8):
        g = torch.Generator(device=dev).manual_seed(100 + K)
        mins = [{"xbc": torch.randn((R, K, shape.cdim), generator=g, device=dev).to(torch.bfloat16),
                 "dt_raw": torch.randn((R, K, shape.nheads), generator=g, device=dev),
                 "z": torch.randn((R, K, shape.nheads * shape.headdim), generator=g,
                                  device=dev).to(torch.bfloat16)} for _ in range(2)]
        yk = torch.empty((R, K, shape.nheads, shape.headdim), dtype=torch.bfloat16, device=dev)
        dk = ssd.dims(R, K, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                      shape.conv_width)

        def kstep(t, mins=mins, yk=yk, dk=dk):
            inp = mins[t % 2]
            ssd.ssd_decode_step(dk, ssd.SSD_BF16, flags, inp["xbc"], prm["conv_w"], prm["conv_b"],
                                pools["conv_pool"], inp["dt_raw"], prm["dt_bias"], prm["A"],
                                prm["D"], inp["z"], pools["slot_ids"], nslots, pools["ssm_pool"],
                                yk, stream)
        for t in range(3):
            kstep(t)
        torch.cuda.synchronize()
        n = 16
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        queue_ahead(statistics.median(host_s[1:]), n)
        e0.record(stream)
        for t in range(n):
            kstep(t)
        e1.record(stream)
        torch.cuda.synchronize()
        kms = ev_ms = e0.elapsed_time(e1) / n
        multi[f"K{K}"] = {"ms_per_call": round(kms, 5), "tokens_per_s": round(R * K / (kms / 1e3), 1),
                          "state_gbs": round(sb / (kms / 1e3) / 1e9, 1),
                          "vs_K_single_steps": round(K * ms / ev_ms, 2)}
        del mins, yk
    assert ssd.ssd_read_device_error(stream) == ssd.SSD_OK
    return {"metric": "decode-step state GB/s", "value": round(gbs * world, 1), "unit": "GB/s",
            "per_gpu_gbs": round(gbs, 1), "ms_per_step": round(ms, 5), "steps": steps,
            "rows": R, "slots": nslots, "state_bytes_per_step": sb,
            "all_bytes_gbs": round(total, 1), "peak": hbm, "peak_source": src,
            "frac": round(gbs / hbm, 4), "traffic": ncu_traffic("decode"),
            "tokens_per_s": round(R / (ms / 1e3), 1),
            "multi_token": multi}


# ---------------------------------------------------------------------------
# the fp64 oracle on the host cores

def oracle_sample_rows() -> int:
    return int(os.environ.get("SSD_BENCH_ORACLE_ROWS", str(si.LONG.seqlen)))


def oracle_prefill_sample(rows: int):
    """Time the oracle on one sequence of the long workload's first call (its
    first ``rows`` rows, all 128 heads: conv + SiLU + recurrence + gate).  The
    oracle's cost per row does not depend on the sequence or on the row's
    position, so its rate on this sample is its rate on the whole workload.
    Returns (seconds, threads)."""
    import oracle
    import numpy as np
    shape = si.LONG.with_(batch=1, seqlen=rows)
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
    """The oracle on a sample of the long workload, repeated until at least
    `min_seconds` of wall time (at least once)."""
    rows = oracle_sample_rows()
    total, passes, threads = 0.0, 0, 1
    while passes == 0 or total < min_seconds:
        dt, threads = oracle_prefill_sample(rows)
        total += dt
        passes += 1
    rate = rows * passes / total
    step_rows = LONG_STEP.batch * LONG_STEP.seqlen
    return {"value": round(rate, 2), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{passes} passes over one {rows}-row sequence of the long workload's "
                      f"first call, all 128 heads (conv + recurrence + gate, fp64), "
                      f"{total:.1f} s; a whole step ({step_rows} rows) extrapolates to "
                      f"{step_rows / rate:.0f} s"}


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
        "config": {"workload": "nemotron-h-8b mixer long prefill (as the main arm); each step "
                               f"is a bounded sample: one {rows}-row sequence of the first call, "
                               "all 128 heads",
                   "batch_per_gpu": 1, "seq_len": rows, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"one {rows}-row sequence x 128 heads per step"},
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
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the decay-stress, packed-sequence and gated-norm workloads")
    ap.add_argument("--only", choices=["all", "long", "prefill", "decode", "tail", "stress"],
                    default="all",
                    help="time only the long-prefill steps, the 2048-row prefill calls, "
                         "the decode steps, the scan + gated norm calls or the decay-stress "
                         "passes (profiler runs)")
    ap.add_argument("--long-batch", type=int, default=si.LONG.batch,
                    help="sequences of the long workload (8; fewer only to keep profiler "
                         "captures small)")
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
