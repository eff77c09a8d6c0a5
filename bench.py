#!/usr/bin/env python3
"""KDA hot-path benchmark on one GB300 (or N independent replicas under torchrun).

Headline (`value`): prefill tokens/s per layer on the single-request prefill workload (B=1, T=8192, H=12,
d=128, bf16 q/k/v, fp32 gates and state, S0 ~ N(0, 0.02), bf16 outputs + final fp32 state).  One step is
one pass of the prefill path over that batch: the copy-on-write restore of the checkpoint into the working
slot followed by the chunked (or segmented) prefill.  Inputs are resident in HBM; L2 is flushed (a 512 MB
write) between timed steps.

Also reported (`decode_verify`): state GB/s of the decode step, the 8-token speculative verify and the
replay fold on the batched workload (256 requests, 1024-slot pool), against the measured HBM peak; and
(`backward`) the prefill backward (all input and initial-state gradients) on the single-request workload.

`--impl reference` times the fp64 CPU oracle (the baseline arm) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
BYTES_PER_TOKEN_HEAD = 3 * 256 + 512 + 4 + 256  # q, k, v bf16 + g fp32 + beta fp32 in; o bf16 out (d = 128)
STATE_BYTES = 128 * 128 * 4
RECORD_BYTES = 256 + 256 + 512 + 4  # k, v bf16 + g fp32 + beta fp32
# chunk-form algorithmic FLOPs per token and head at d = 128, C = 64: 2 (3 d^2 + 2.5 C d + C^2 / 6)
ALG_FLOP_PER_TOKEN_HEAD = 2 * (3 * 128 * 128 + 2.5 * 64 * 128 + 64 * 64 / 6)
# DRAM traffic per launch of a kernel, from one ncu capture, keyed by the SHA-256 of the kernel's source
# files: reported as the roofline's traffic only while the committed sources still hash to that value
TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
CSRC = os.path.join(ROOT, "kda_gated_delta_rule_gb300", "csrc")


def source_sha256(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str, table: str = TRAFFIC_TABLE):
    """DRAM bytes (read + write) of one launch of `kernel` on `workload` from the traffic table, or None when
    the table has no row for it or the kernel's sources changed since the capture."""
    if not os.path.exists(table):
        return None
    for line in open(table):
        if not line.strip() or line.startswith("#"):
            continue
        f = line.rstrip("\n").split("\t")
        if len(f) < 6 or f[0] != kernel or f[1] != workload:
            continue
        try:
            if source_sha256(f[2].split(",")) != f[3]:
                return None
        except OSError:
            return None
        return int(f[4]) + int(f[5])
    return None


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine() or "unknown"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--path", choices=["auto", "varlen", "segmented"], default="segmented")
    ap.add_argument("--segment-len", type=int, default=0,
                    help="tokens per segment of the segmented path (multiple of 64); 0 = the shortest segment whose "
                         "output phase (one CTA per head and segment) fits one wave on this GPU")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode/verify/fold measurements")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward measurement")
    ap.add_argument("--no-cfbi", action="store_true", help="skip the batch-invariant prefill measurement")
    ap.add_argument("--no-varlen", action="store_true", help="skip the varlen packed-prefill workload")
    ap.add_argument("--no-long", action="store_true", help="skip the 1M-token segmented prefill workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Weak scaling: every rank processes its own copy of the workload; the job rate is the units of all
    ranks over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ---------------------------------------------------------------- clocks

class Clocks:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            if self.uuid and self.uuid not in parts[0]:
                continue
            rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- our arm

def run_ours(args):
    import torch

    import kda_gated_delta_rule_gb300 as kda

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    kda.load()
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "")) or None
    if uuid and not uuid.startswith("GPU-"):
        uuid = "GPU-" + uuid
    pk, pk_kind = peaks()
    stream = torch.cuda.current_stream()

    def to_dev(x):
        t = torch.from_numpy(np.ascontiguousarray(x))
        return (t.view(torch.bfloat16) if x.dtype == np.uint16 else t).to(dev)

    # ---- single-request prefill workload
    prob = synth.prefill_8k()
    T, H, d = prob.T, prob.H, prob.dk
    q, k, v, g, beta = (to_dev(x) for x in (prob.q, prob.k, prob.v, prob.g, prob.beta))
    cu = to_dev(prob.cu_seqlens.astype(np.int32))
    ckpt = to_dev(prob.pool)              # the checkpoint (committed prefix state)
    pool = torch.zeros_like(ckpt)         # the working slot
    slot = to_dev(np.array([0], np.int32))
    out = torch.empty(T, H, d, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(2, dtype=torch.int32, device=dev)
    pargs = (q, k, v, g, beta, cu, T, pool, slot, out)
    if args.segment_len > 0:
        seg_candidates = [args.segment_len]
    else:
        # segment lengths from one output-phase CTA per SM and head (H CTAs per segment) down to about half
        # as many segments; the fastest on a few untimed steps is taken
        one_wave = max(1, props.multi_processor_count // H)
        ceil_div = lambda x, y: -(-x // y)
        seg_candidates = sorted({64 * ceil_div(ceil_div(T, P), 64) for P in range(max(1, one_wave // 2), one_wave + 2)})
    ws_bytes = max(kda.kda_segmented_workspace_size(*pargs, sl) for sl in seg_candidates)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    ws_var = torch.empty(max(kda.kda_prefill_workspace_size(*pargs), 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def restore():
        kda.kda_state_copy(ckpt, slot, pool, slot)

    def prefill(path, sl=None):
        if path == "varlen":
            kda.kda_prefill_varlen(*pargs, workspace=ws_var, dev_status=status)
        else:
            kda.kda_prefill_segmented(*pargs, sl, ws, dev_status=status)

    kernels_per_step = {"varlen": 3, "segmented": 5}  # state copy + the path's kernels

    def time_calls(fn, n, flush_between=True):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            if flush_between:
                flush.zero_()
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    # choose the path and segment length (all are parity-tested): the fastest on a few untimed calls
    paths = ["varlen", "segmented"] if args.path == "auto" else [args.path]
    trial = {}
    for pth in paths:
        for sl in (seg_candidates if pth == "segmented" else [None]):
            for _ in range(2):
                restore()
                prefill(pth, sl)
            torch.cuda.synchronize()
            trial[(pth, sl)] = statistics.median(time_calls(lambda: (restore(), prefill(pth, sl)), 5))
    path, seg_len = min(trial, key=trial.get)

    # the step's launches, phase by phase (exactly the kernels kda_prefill_varlen / kda_prefill_segmented
    # enqueue), so the timed steps also give each kernel's duration from events between its launches
    if path == "varlen":
        phase_fns = [("kda_state_copy", restore),
                     ("tc_prep_kernel", lambda: kda.kda_prefill_records(*pargs, workspace=ws_var, dev_status=status)),
                     ("tc_chain_kernel<plain>",
                      lambda: kda.kda_prefill_chain(*pargs, workspace=ws_var, dev_status=status))]
    else:
        phase_fns = [("kda_state_copy", restore),
                     ("tc_prep_kernel", lambda: kda.kda_prefill_records(*pargs, workspace=ws, dev_status=status)),
                     ("tc_chain_kernel<frag>",
                      lambda: kda.kda_segment_fragments(*pargs, seg_len, ws, dev_status=status)),
                     ("seg_scan_kernel", lambda: kda.kda_fragment_scan(*pargs, seg_len, ws, dev_status=status)),
                     ("tc_chain_kernel<segout>",
                      lambda: kda.kda_segment_outputs(*pargs, seg_len, ws, dev_status=status))]

    def step():
        for _, fn in phase_fns:
            fn()

    def time_steps(n, phases=False):
        # events around every step; with `phases`, also between its kernels (an event between two kernels
        # holds the second back until the first has finished, so the step times are taken without them)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(phase_fns) + 1)] for _ in range(n)]
        for i in range(n):
            flush.zero_()
            evs[i][0].record(stream)
            for j, (_, fn) in enumerate(phase_fns):
                fn()
                if phases or j + 1 == len(phase_fns):
                    evs[i][j + 1].record(stream)
        torch.cuda.synchronize()
        steps_ms = [e[0].elapsed_time(e[-1]) for e in evs]
        per_phase = {name: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n))
                     for j, (name, _) in enumerate(phase_fns)} if phases else None
        return steps_ms, per_phase

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    status.zero_()

    clocks = Clocks(uuid).start()
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    step_ms, _ = time_steps(args.steps)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    # per-kernel durations: the same steps again, with an event between their kernels
    phase_step_ms, phases = time_steps(args.steps, phases=True)
    clk = clocks.stop()
    st = status.cpu().numpy()
    if st[0] != 0 or st[1] == 0:
        raise RuntimeError(f"device status {st.tolist()} after the timed region (flags set or no work done)")
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, world, dev)
    value = whole_job_value(T, world, ms_max / 1e3)

    # ---- per-kernel durations: events between the launches of a second pass of the timed steps (above)
    dominant = max((kname for kname in phases if kname != "kda_state_copy"), key=lambda kname: phases[kname])
    # algorithmic bytes of the prefill: 1540 B per token and head (q, k, v, o bf16; g, beta fp32) plus the
    # initial and final state of every head; achieved = those bytes / the dominant kernel's duration
    alg_bytes = T * H * BYTES_PER_TOKEN_HEAD + 2 * H * STATE_BYTES
    achieved = alg_bytes / (phases[dominant] / 1e3) / 1e9
    path_gbs = alg_bytes / (ms_max / 1e3) / 1e9
    roofline = {"kernel": dominant, "bound": "hbm", "achieved": round(achieved, 2), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 5),
                "traffic": measured_traffic(dominant, "prefill_8k"),
                "peak_source": pk_kind, "algorithmic_bytes": alg_bytes,
                "kernel_ms": round(phases[dominant], 4),
                "phase_ms": {kk: round(vv, 4) for kk, vv in phases.items()},
                "phase_pass_ms_per_step": round(statistics.mean(phase_step_ms), 4),
                "step_gbs": round(path_gbs, 2), "step_frac": round(path_gbs / pk["hbm_gbs"], 5),
                "algorithmic_tflops_step": round(T * H * ALG_FLOP_PER_TOKEN_HEAD / (ms_max / 1e3) / 1e12, 3)}

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region
    hq, hk, hv, hg, hb = (torch.from_numpy(np.ascontiguousarray(x)).pin_memory() for x in
                          (prob.q, prob.k, prob.v, prob.g, prob.beta))
    hs0 = torch.from_numpy(prob.pool).pin_memory()
    ho = torch.empty(T, H, d, dtype=torch.bfloat16).pin_memory()
    hsf = torch.empty_like(hs0).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hg, hb, hs0))
    d2h = ho.numel() * ho.element_size() + hsf.numel() * hsf.element_size()

    # Steps are pipelined over three streams (host->device, compute, device->host) with double-buffered device
    # inputs and outputs, so step k+1's inputs upload while step k computes; every step still carries its own
    # copies.  L2 is flushed on the compute stream before each step's kernels.
    sets = []
    for _ in range(2):
        sets.append({"x": [torch.empty_like(t) for t in (q, k, v, g, beta)], "ckpt": torch.empty_like(ckpt),
                     "pool": torch.empty_like(pool), "out": torch.empty_like(out)})
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(n):
        ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(n)] for _ in range(3))
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t_start.record(s_in)
        for i in range(n):
            st = sets[i % 2]
            dx = st["x"]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[i - 2])  # this set's inputs were consumed by step i - 2
                for dst, src in zip(dx, (hq, hk, hv, hg, hb)):
                    if dst.dtype == torch.bfloat16:  # host bf16 inputs are held as raw 16-bit words
                        dst.view(torch.int16).copy_(src.view(torch.int16), non_blocking=True)
                    else:
                        dst.copy_(src, non_blocking=True)
                st["ckpt"].copy_(hs0, non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[i])
                if i >= 2:
                    s_cmp.wait_event(ev_out[i - 2])  # this set's outputs were read back
                flush.zero_()
                kda.kda_state_copy(st["ckpt"], slot, st["pool"], slot)
                eargs = (*dx, cu, T, st["pool"], slot, st["out"])
                if path == "varlen":
                    kda.kda_prefill_varlen(*eargs, workspace=ws_var, dev_status=status)
                else:
                    kda.kda_prefill_segmented(*eargs, seg_len, ws, dev_status=status)
                ev_cmp[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[i])
                ho.copy_(st["out"], non_blocking=True)
                hsf.copy_(st["pool"], non_blocking=True)
                ev_out[i].record(s_out)
        t_end.record(s_out)
        torch.cuda.synchronize()
        return t_start.elapsed_time(t_end) / n

    e2e_run(3)
    e2e_steps = max(5, min(args.steps, 20))
    e2e_ms = e2e_run(e2e_steps)
    if not torch.equal(ho.view(torch.int16), out.view(torch.int16).cpu()):  # same inputs, same kernels: same bits
        raise RuntimeError("the end-to-end outputs differ from the device-resident run's")
    e2e_value = whole_job_value(T, world, max_over_ranks(e2e_ms, world, dev) / 1e3)

    # ---- decode / verify / fold on the batched workload
    dv_report = None
    if not args.no_decode:
        dv_report = decode_verify_report(kda, torch, dev, to_dev, time_calls, pk, world)

    bw_report = None
    if not args.no_backward:
        bw_report = backward_report(kda, torch, dev, to_dev, time_calls, pk, prob)

    cf_report = None
    if not args.no_cfbi:
        cf_report = cfbi_prefill_report(kda, torch, dev, to_dev, time_calls, pk, prob)

    # ---- the varlen packed prefill and the 1M-token segmented prefill (tokens/s, fraction of HBM)
    del ws, ws_var, sets
    torch.cuda.empty_cache()
    with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    varlen_report = long_report = None
    if not args.no_varlen:
        vprob = synth.varlen()
        varlen_report = prefill_workload_report(
            kda, torch, dev, to_dev, vprob, varlen_candidates(vprob, props.multi_processor_count),
            steps=max(5, min(args.steps, 20)), warmup=args.warmup, pk=pk, oracle_tokens=16384, oracle_seconds=5.0,
            with_cpu=with_cpu)
        varlen_report["workload"] = ("varlen packed prefill: 16 sequences, lengths log-uniform in [512, 32768] "
                                     f"({vprob.T} tokens), H=12, d=128, bf16 q/k/v, 256-slot fp32 pool gathered and "
                                     "scattered by slot id, snapshots every 4 chunks into a ping-pong extra pool")
        del vprob
    if not args.no_long:
        lprob = synth.long_1m()
        long_report = prefill_workload_report(
            kda, torch, dev, to_dev, lprob, [("segmented", lprob.segment_len)], steps=5, warmup=2, pk=pk,
            oracle_tokens=16384, oracle_seconds=5.0, with_cpu=with_cpu)
        long_report["workload"] = ("long-context prefill: B=1, T=1,048,576, H=12, d=128, bf16 q/k/v, fp32 gates and "
                                   "state, 64 segments of 16,384 tokens composed by the on-GPU fragment scan")
        del lprob

    line = {
        "metric": "KDA prefill tokens/s/layer (H=12,d=128); decode+verify state GB/s vs HBM peak",
        "value": round(value, 1),
        "unit": "tokens/s/layer",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16x3",
        "data": "synthetic",
        "config": {
            "workload": "single-request prefill: B=1, T=8192, H=12, dk=dv=128, bf16 q/k/v, fp32 g/beta, "
                        "fp32 state S0~N(0,0.02), bf16 o + final fp32 state; step = COW restore + prefill",
            "path": path, "segment_len": seg_len if path == "segmented" else None,
            "path_trial_ms": {(f"{kk[0]}/{kk[1]}" if kk[1] else kk[0]): round(vv, 4) for kk, vv in trial.items()},
            "l2": "flushed between timed steps (512 MB write)",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
        },
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s/layer", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "pipeline": "host->device, compute and device->host streams, two device buffer sets; L2 flushed "
                            "on the compute stream before each step"},
        "gpu_launches": args.steps * kernels_per_step[path],
        "clocks": clk,
        "wall_s_timed_region": round(wall, 4),
    }
    if dv_report:
        line["decode_verify"] = dv_report
    if bw_report:
        line["backward"] = bw_report
    if cf_report:
        line["cfbi_prefill"] = cf_report
    if varlen_report:
        line["varlen_prefill"] = varlen_report
    if long_report:
        line["long_prefill"] = long_report
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(prob, sample_tokens=T)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def decode_verify_report(kda, torch, dev, to_dev, time_calls, pk, world):
    p = synth.decode_verify()
    B, W, H, d = p.B, p.W, p.H, p.dk
    pool = to_dev(p.pool)
    slots = to_dev(p.slot_ids)
    q, k, v, g, beta = (to_dev(x) for x in (p.q, p.k, p.v, p.g, p.beta))
    wq, wk, wv, wg, wb = (to_dev(x) for x in (p.wq, p.wk, p.wv, p.wg, p.wbeta))
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    wout = torch.empty(B, W, H, d, dtype=torch.bfloat16, device=dev)
    rec = torch.empty(kda.kda_replay_bytes(B, W, H, d, d, p.in_dtype), dtype=torch.uint8, device=dev)
    acc = to_dev(p.accepted)
    # checkpoint slots drawn from the slots the requests do not hold: a copy's source and destination never alias
    free = np.setdiff1d(np.arange(p.pool.shape[0], dtype=np.int32), p.slot_ids)
    ckpt_slots = to_dev(free[synth.distinct_slots(p.seed, 99, B, free.size)].astype(np.int32))

    def dec():
        kda.kda_decode_step(q, k, v, g, beta, pool, slots, out)

    def ver():
        kda.kda_verify(wq, wk, wv, wg, wb, pool, slots, wout, rec)

    def fold():
        kda.kda_verify_replay(pool, slots, rec, acc, W, H, d, d, p.in_dtype)

    def copy():
        kda.kda_state_copy(pool, ckpt_slots, pool, slots)

    # CF-BI decode: open-chunk row counts uniform in [0, 16) (seeded), row caches in their own pool
    CH, RF = kda.CFBI_CHUNK, kda.CFBI_ROW_FLOATS
    n_open = (synth.uniform(p.seed, 98, p.pool.shape[0] * H) * CH).astype(np.int32).reshape(p.pool.shape[0], H)
    counts0 = to_dev(np.minimum(n_open, CH - 1))
    cache = torch.zeros(p.pool.shape[0], H, CH, RF, dtype=torch.float32, device=dev)
    cache[..., 256:384] = -0.1 * torch.arange(CH, device=dev, dtype=torch.float32).view(1, 1, CH, 1)
    counts = counts0.clone()
    cf_out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)

    def cfbi():
        counts.copy_(counts0)  # the same open-chunk positions every call (a 1.5 MB copy, timed with it)
        kda.kda_cfbi_decode(q, k, v, g, beta, pool, cache, counts, slots, cf_out)

    # fused decode (short convolution + KDA step + gated output norm) on the same pool and slots
    fz = synth.fused_decode_inputs(p.seed, B, H, d, p.pool.shape[0], 1, p.in_dtype, with_pool=False)
    fx = [to_dev(fz[nm][0]) for nm in ("xq", "xk", "xv", "a", "b", "z")]
    fcs, fcw, fnw = to_dev(fz["conv_state"]), to_dev(fz["conv_w"]), to_dev(fz["norm_w"])
    f_out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)

    def fused():
        kda.kda_fused_decode(*fx, pool, slots, fcs, fcw, fnw, f_out)

    for fn in (dec, ver, fold, copy, cfbi, fused):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    n = 20
    runs = {name: time_calls(fn, n) for name, fn in
            (("decode", dec), ("verify", ver), ("fold", fold), ("state_copy", copy), ("cfbi_decode", cfbi),
             ("fused_decode", fused))}
    t = {name: statistics.mean(v) for name, v in runs.items()}
    heads = B * H
    n_acc = p.accepted.astype(np.int64)
    alg = {
        "decode": heads * (2 * STATE_BYTES + BYTES_PER_TOKEN_HEAD),
        "verify": heads * (STATE_BYTES + W * (BYTES_PER_TOKEN_HEAD + RECORD_BYTES)),
        "fold": int(H * sum(2 * STATE_BYTES + nn * RECORD_BYTES for nn in n_acc if nn > 0)),
        "state_copy": B * 2 * H * STATE_BYTES,
        # entry state read, L cached rows read, then the new row written (or, completing a chunk, the state
        # written), plus the token's inputs and output
        "cfbi_decode": int(sum(STATE_BYTES + BYTES_PER_TOKEN_HEAD + nl * RF * 4 + (RF * 4 if nl < CH - 1 else STATE_BYTES)
                               for nl in np.minimum(n_open, CH - 1)[p.slot_ids].ravel())),
        # state and carried convolution inputs (3 streams x 3 taps x d fp32) read and written; xq, xk, xv, z
        # bf16, a fp32, b in; out bf16
        "fused_decode": heads * (2 * STATE_BYTES + 2 * 9 * d * 4 + 4 * 2 * d + 4 * d + 4 + 2 * d),
    }
    rep = {"workload": "batched decode + speculative verify: 256 requests, 1024-slot pool, H=12, d=128, "
                       "W=8, accepted ~ min(Poisson(2.7), 8)", "peak_gbs": pk["hbm_gbs"],
           "timing": f"{n} calls each, L2 flushed before every call; ms = mean, ms_median = median"}
    for name in t:
        gbs = alg[name] / (t[name] / 1e3) / 1e9
        med = statistics.median(runs[name])
        rep[name] = {"ms": round(t[name], 5), "algorithmic_bytes": alg[name], "gbs": round(gbs, 1),
                     "frac": round(gbs / pk["hbm_gbs"], 4), "ms_median": round(med, 5),
                     "frac_median": round(alg[name] / (med / 1e3) / 1e9 / pk["hbm_gbs"], 4)}
    return rep


def prefill_workload_report(kda, torch, dev, to_dev, prob, candidates, steps, warmup, pk, oracle_tokens,
                            oracle_seconds, with_cpu):
    """Tokens/s of one packed prefill workload on the device: each step restores the sequences' initial
    states from a checkpoint pool (a state copy of N slots) and runs the prefill over the whole batch
    (gather from the pool, chunk path, snapshots, scatter back).  `candidates` are (path, segment length)
    pairs, each timed over a few untimed steps; the fastest is timed over `steps`.  The inputs are larger
    than L2, so no flush between steps.  Algorithmic bytes: 1540 per token and head, the initial and final
    state of every (sequence, head), and the snapshot states left in the extra pool."""
    T, H, d, N = prob.T, prob.H, prob.dk, prob.N
    q, k, v, g, beta = (to_dev(x) for x in (prob.q, prob.k, prob.v, prob.g, prob.beta))
    cu = to_dev(prob.cu_seqlens.astype(np.int32))
    ckpt = to_dev(prob.pool)
    pool = ckpt.clone()
    slots = to_dev(prob.slot_ids.astype(np.int32))
    out = torch.empty(T, H, d, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(2, dtype=torch.int32, device=dev)
    max_len = int(prob.lengths.max())
    common = {}
    every = 0
    if prob.extra_pool is not None and prob.snapshot_every_chunks:
        common = dict(extra_pool=to_dev(prob.extra_pool), extra_slot_ids=to_dev(prob.extra_slot_ids.astype(np.int32)),
                      snapshot_every_chunks=prob.snapshot_every_chunks)
        every = 64 * prob.snapshot_every_chunks
    pargs = (q, k, v, g, beta, cu, max_len, pool, slots, out)

    def restore():
        kda.kda_state_copy(ckpt, slots, pool, slots)

    def make(path, seg):
        if path == "varlen":
            ws = torch.empty(max(kda.kda_prefill_workspace_size(*pargs, **common), 256), dtype=torch.uint8, device=dev)
            return ws, lambda: kda.kda_prefill_varlen(*pargs, workspace=ws, dev_status=status, **common)
        ws = torch.empty(max(kda.kda_segmented_workspace_size(*pargs, seg, **common), 256), dtype=torch.uint8,
                         device=dev)
        return ws, lambda: kda.kda_prefill_segmented(*pargs, seg, ws, dev_status=status, **common)

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            a.record()
            restore()
            fn()
            b.record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    trial = {}
    for path, seg in candidates:
        ws, fn = make(path, seg)
        timed(fn, 1)
        trial[(path, seg)] = statistics.median(timed(fn, 2))
        del ws, fn
        torch.cuda.empty_cache()
    path, seg = min(trial, key=trial.get)
    ws, fn = make(path, seg)
    timed(fn, max(warmup, 3))
    status.zero_()
    step_ms = statistics.mean(timed(fn, steps))
    st = status.cpu().numpy()
    if st[0] != 0 or st[1] == 0:
        raise RuntimeError(f"{prob.name}: device status {st.tolist()} (flags set or no work done)")
    n_snapshots = sum(min(int(n) // every, 2) for n in prob.lengths) if every else 0
    alg = T * H * BYTES_PER_TOKEN_HEAD + 2 * N * H * STATE_BYTES + n_snapshots * H * STATE_BYTES
    gbs = alg / (step_ms / 1e3) / 1e9
    rep = {"tokens": T, "sequences": N, "path": path, "segment_len": seg if path == "segmented" else None,
           "path_trial_ms": {f"{pp}/{sg}" if pp == "segmented" else pp: round(tt, 4) for (pp, sg), tt in trial.items()},
           "steps": steps, "ms_per_step": round(step_ms, 4), "tokens_per_s": round(T / (step_ms / 1e3), 1),
           "algorithmic_bytes": alg, "gbs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 5),
           "algorithmic_tflops": round(T * H * ALG_FLOP_PER_TOKEN_HEAD / (step_ms / 1e3) / 1e12, 3),
           "l2": "inputs larger than L2 (no flush)", "step": "state restore of the N slots + prefill"}
    if every:
        rep["snapshot_states_written"] = n_snapshots * H
        rep["snapshot_note"] = (f"only the last two snapshots of each sequence survive the call and only they are "
                                f"written: {n_snapshots * H * STATE_BYTES} B; writing every one of the "
                                f"{sum(int(n) // every for n in prob.lengths) * H} snapshot states would add "
                                f"{(sum(int(n) // every for n in prob.lengths) - n_snapshots) * H * STATE_BYTES} B")
    del ws, fn
    torch.cuda.empty_cache()
    if with_cpu:
        rep["cpu_baseline"] = cpu_baseline(prob, sample_tokens=oracle_tokens, min_seconds=oracle_seconds,
                                           snap_every=every)
    return rep


def varlen_candidates(prob, sms):
    """The varlen path (one chain per sequence and head) and the segmented path at segment lengths around the
    one that spreads the token-heads evenly over one CTA per SM."""
    even = max(64, -(-int(prob.T) * prob.H // (sms * prob.H)) // 64 * 64)
    segs = sorted({max(256, s // 64 * 64) for s in (even // 2, even, 2 * even, 4 * even)})
    return [("varlen", 0)] + [("segmented", s) for s in segs]


# gradient bytes per token and head of the backward: q, k, v, d_out bf16 + g, beta fp32 in; dq, dk, dv, dg, dbeta
# fp32 out (d = 128)
BW_BYTES_PER_TOKEN_HEAD = 4 * 256 + 512 + 4 + 4 * 512 + 4


def backward_report(kda, torch, dev, to_dev, time_calls, pk, prob):
    """The prefill backward on the single-request workload: one call = all six kernels."""
    T, H, N = prob.T, prob.H, prob.N
    d_out, d_final = synth.output_grads(prob, prob.seed)
    q, k, v, g, beta, dout = (to_dev(x) for x in (prob.q, prob.k, prob.v, prob.g, prob.beta, d_out))
    dfin = to_dev(d_final)
    cu = to_dev(prob.cu_seqlens.astype(np.int32))
    pool, slots = to_dev(prob.pool), to_dev(prob.slot_ids)
    grads = [torch.empty(T, H, 128, device=dev) for _ in range(4)]
    dbeta = torch.empty(T, H, device=dev)
    dinit = torch.empty(N, H, 128, 128, device=dev)
    ws = torch.empty(kda.kda_backward_workspace_size(T, N, H), dtype=torch.uint8, device=dev)
    max_len = int(prob.lengths.max())

    def call():
        kda.kda_prefill_backward(q, k, v, g, beta, cu, max_len, dout, *grads, dbeta, ws, pool=pool, slot_ids=slots,
                                 d_final=dfin, d_init=dinit)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ms = statistics.mean(time_calls(call, 20))
    alg = T * H * BW_BYTES_PER_TOKEN_HEAD + N * H * 3 * STATE_BYTES
    gbs = alg / (ms / 1e3) / 1e9
    return {"workload": "prefill backward: B=1, T=8192, H=12, d=128, bf16 q/k/v/d_out, fp32 gradients out, "
                        "S0 and dL/dS_T given, dL/dS0 out; L2 flushed between calls",
            "ms": round(ms, 4), "tokens_per_s": round(T / (ms / 1e3), 1), "algorithmic_bytes": alg,
            "gbs": round(gbs, 1), "frac": round(gbs / pk["hbm_gbs"], 4), "kernels_per_call": 13,
            "workspace_bytes": ws.numel()}


def cfbi_prefill_report(kda, torch, dev, to_dev, time_calls, pk, prob):
    """The batch-invariant (CF-BI) prefill on the single-request workload: the chunk-parallel call (rows, then
    the state walk; one call = two kernels) and, for reference, the token-sequential call, which must give
    the same bits.  Each call first restores the pool and zeroes the row counts (a 6 MB copy and a memset,
    timed with the call)."""
    T, H, N = prob.T, prob.H, prob.N
    q, k, v, g, beta = (to_dev(x) for x in (prob.q, prob.k, prob.v, prob.g, prob.beta))
    cu = to_dev(prob.cu_seqlens.astype(np.int32))
    pool0, slots = to_dev(prob.pool), to_dev(prob.slot_ids)
    pool = pool0.clone()
    cache = torch.zeros(prob.pool.shape[0], H, kda.CFBI_CHUNK, kda.CFBI_ROW_FLOATS, device=dev)
    counts = torch.zeros(prob.pool.shape[0], H, dtype=torch.int32, device=dev)
    out = torch.empty(T, H, 128, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(kda.kda_cfbi_prefill_chunked_workspace_size(T, N, H), dtype=torch.uint8, device=dev)
    max_len = int(prob.lengths.max())

    def chunked():
        pool.copy_(pool0)
        counts.zero_()
        kda.kda_cfbi_prefill_chunked(q, k, v, g, beta, cu, max_len, pool, cache, counts, slots, out, ws)

    def sequential():
        pool.copy_(pool0)
        counts.zero_()
        kda.kda_cfbi_prefill(q, k, v, g, beta, cu, max_len, pool, cache, counts, slots, out)

    for _ in range(3):
        chunked()
    torch.cuda.synchronize()
    ms = statistics.mean(time_calls(chunked, 10))
    o_chunked, p_chunked = out.clone(), pool.clone()
    ms_seq = statistics.mean(time_calls(sequential, 2))
    same = bool(torch.equal(o_chunked, out) and torch.equal(p_chunked, pool))
    if not same:
        raise RuntimeError("the chunk-parallel CF-BI prefill differs from the token-sequential one")
    alg = T * H * BYTES_PER_TOKEN_HEAD + 2 * N * H * STATE_BYTES
    gbs = alg / (ms / 1e3) / 1e9
    return {"workload": "batch-invariant (CF-BI, 16-token chunks) prefill: B=1, T=8192, H=12, d=128, bf16 q/k/v, "
                        "fp32 gates and state, bf16 o; fresh open chunk; L2 flushed between calls",
            "ms": round(ms, 4), "tokens_per_s": round(T / (ms / 1e3), 1), "algorithmic_bytes": alg,
            "gbs": round(gbs, 1), "frac": round(gbs / pk["hbm_gbs"], 4), "kernels_per_call": 2,
            "workspace_bytes": ws.numel(), "token_sequential_ms": round(ms_seq, 3),
            "bit_identical_to_token_sequential": same}


# ---------------------------------------------------------------- CPU baseline (the oracle)

def cpu_baseline(prob, sample_tokens, min_seconds=10.0, max_repeats=2000, snap_every=0):
    """The oracle as it stands, timed on the host cores over the sample (the first `sample_tokens` tokens of
    the longest sequence), repeated until about `min_seconds` of work have been timed; value = tokens
    processed / seconds."""
    import oracle
    i = int(np.argmax(prob.lengths))
    a = int(prob.cu_seqlens[i])
    sample_tokens = min(sample_tokens, int(prob.lengths[i]))
    q, k, v, g, beta = (x[a:a + sample_tokens] for x in (prob.q, prob.k, prob.v, prob.g, prob.beta))
    s0 = prob.pool[prob.slot_ids[i:i + 1]].astype(np.float64)
    reps = 0
    t0 = time.perf_counter()
    while True:
        r = oracle.recurrence(q, k, v, g, beta, [0, sample_tokens], s0=s0, snap_every=snap_every)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or reps >= max_repeats:
            break
    return {"value": round(reps * sample_tokens / dt, 2), "unit": "tokens/s/layer", "cores": r["threads"],
            "cpu_model": cpu_model(), "kind": "oracle", "seconds": round(dt, 3), "repeats": reps,
            "sample": f"first {sample_tokens} tokens x {prob.H} heads of the longest sequence of the {prob.name} workload (fp64 "
                      f"sequential recurrence, all outputs + final state"
                      f"{', snapshots every %d tokens' % snap_every if snap_every else ''}), {reps} passes in "
                      f"{dt:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    prob = synth.prefill_8k()
    sample = 2048
    q, k, v, g, beta = (x[:sample] for x in (prob.q, prob.k, prob.v, prob.g, prob.beta))
    s0 = prob.pool[prob.slot_ids].astype(np.float64)

    def step():
        return oracle.recurrence(q, k, v, g, beta, [0, sample], s0=s0)

    for _ in range(max(args.warmup, 3)):
        r = step()
    times = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    wall = time.perf_counter() - t_all
    s = statistics.mean(times)
    value = sample / s
    line = {
        "impl": "reference",
        "metric": "KDA prefill tokens/s/layer (H=12,d=128); decode+verify state GB/s vs HBM peak",
        "value": round(value, 2), "unit": "tokens/s/layer", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "single-request prefill: B=1, T=8192, H=12, dk=dv=128 (bounded sample: first "
                               f"{sample} tokens per step)", "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s/layer", "cores": r["threads"],
                         "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": f"first {sample} tokens x 12 heads per step"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s/layer", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s_timed_region": round(wall, 3),
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus > 1 and world == 1 and "LOCAL_RANK" not in os.environ:
        # --gpus N without a launcher: start N ranks on this node (one per GPU) and exit with their status
        import socket
        with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
        sys.exit(subprocess.call(cmd))
    if world != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} but the launcher started {world} rank(s)")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
