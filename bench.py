"""Benchmark: raw-input parse throughput of libpp on one GB300 and its HBM
roofline fraction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one pass of the whole parse hot path (pp_parse: context
identification, tagging, record/column indexing, columnar output, numeric
conversion; or pp_tokenize for the token-stream workload) over one
synthetic input already resident in device memory.  Inputs are larger than
the 129 MB L2, so no flush is needed between steps.  For N > 1 (one process
per GPU, launched by torch.distributed.run) every rank parses its own
replica of the input: the path does not shard, so the scaling is weak and
no data-path collective exists.  Rank 0 prints one JSON line.

--impl reference times the CPU oracle (the plain sequential parser) on this
host's cores, on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import datagen  # noqa: E402

METRIC = "raw-input parse GB/s on 1 GB300 and % of HBM-bandwidth roofline"
DEFAULT_WORKLOAD = "csv18_2gib"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, torch copy)"
    return 6800.0, "fallback (6.8 TB/s earlier GB300 measurement)"


def code_sha(path):
    """sha256 prefix of a CUDA source's code: comments removed and whitespace
    collapsed, so an edit of comments alone leaves it unchanged."""
    import hashlib
    import re
    with open(path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()[:16]


def _traffic(workload):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    capture (profiles/ncu_traffic.json), or None when there is none or the
    kernel's code has changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e:
        return None
    src = os.path.join(ROOT, "dfa_parsing_delimiter_gb300", "csrc",
                       e.get("kernel_source", "pp_parse.cu"))
    if e.get("kernel_code_sha256_prefix") != code_sha(src):
        return None
    return e.get("dram_bytes_per_launch")


class Clocks:
    """Sample nvidia-smi clocks and throttle reasons while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def _max_over_ranks(x, ws, dev):
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _generate_pinned(workload, target=None, record_offsets=False):
    w = datagen.WORKLOADS[workload]
    cap = w["target"] if target is None else target
    h = torch.empty(cap, dtype=torch.uint8, pin_memory=True)
    data, info, _ = datagen.generate(workload, target=cap, out_ptr=h.data_ptr(), out_cap=cap,
                                     record_offsets=record_offsets)
    return h[: info["n_bytes"]], info


def _cpu_baseline(workload, h_in, info, seconds=10.0):
    """Time the oracle on a bounded prefix of the workload (whole records)."""
    import oracle
    w = datagen.WORKLOADS[workload]
    arr = h_in.numpy()
    cores = 1

    def run(nb):
        sample = arr[:nb]
        if w["kind"] == "csv":
            (_, st), dt = oracle.timed_csv_parse(sample, w["cols"])
        else:
            (_, st), dt = oracle.timed_tokenize(sample)
        return dt

    # cut samples at record starts so the sample is whole records
    probe = min(arr.size, 16 << 20)
    dt = run(probe)
    rate = probe / max(dt, 1e-9)
    nb = int(min(arr.size, rate * seconds))
    if w["kind"] == "csv":
        nl = np.flatnonzero(arr[:nb] == 10)
        nb = int(nl[-1]) + 1 if nl.size else nb
    dt = run(nb)
    return {"value": nb / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {nb} bytes of {workload} (whole records), single-threaded "
                      f"sequential DFA walk, parse only, input in RAM",
            "seconds": dt, "host": _cpu_model()}


def _cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part", "hardware")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    w = datagen.WORKLOADS[args.workload]
    h_in, info = _generate_pinned(args.workload)
    import oracle
    arr = h_in.numpy()
    # one bounded sample per step, sized so the whole run takes a few minutes
    probe = min(arr.size, 8 << 20)
    t0 = time.perf_counter()
    if w["kind"] == "csv":
        oracle.csv_parse(arr[:probe], w["cols"])
    else:
        oracle.tokenize(arr[:probe])
    rate = probe / max(time.perf_counter() - t0, 1e-9)
    # about 2.5 minutes of oracle work for the whole run, 0.5 to 4 s a step
    per_step = max(0.5, min(4.0, 150.0 / (args.warmup + args.steps)))
    nb = int(min(arr.size, rate * per_step))
    if w["kind"] == "csv":
        nl = np.flatnonzero(arr[:nb] == 10)
        nb = int(nl[-1]) + 1 if nl.size else nb
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        if w["kind"] == "csv":
            oracle.csv_parse(arr[:nb], w["cols"])
        else:
            oracle.tokenize(arr[:nb])
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = nb * len(times) / tot / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot / len(times) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": args.workload, "n_bytes_sample": nb},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {nb} bytes of {args.workload} per step",
                         "host": _cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure(pp, workload, args, dev, ws, clock_index):
    """Time `args.steps` calls of the hot path on one workload; returns the
    fields of its JSON record (rank 0 adds the CPU baseline)."""
    w = datagen.WORKLOADS[workload]
    h_in, info = _generate_pinned(workload, target=args.target)
    n = int(h_in.numel())
    off = getattr(args, "in_offset", 0)  # bytes past a 256-byte aligned allocation
    d_in = torch.empty(n + 16 + off, dtype=torch.uint8, device=dev)[off:off + n]
    d_in.copy_(h_in)
    stream = torch.cuda.current_stream(dev)
    csv = w["kind"] == "csv"

    if csv:
        desc = pp.desc_csv()
        R = info["n_records"]
        chars_cap = [info["col_value_bytes"][c] if t == "str" else 0
                     for c, t in enumerate(w["cols"])]
        out = pp.CsvOutputs(w["cols"], R, chars_cap, device=dev)

        def step():
            out.run(d_in, n, desc, stream)
        # init, tile vectors, tile states, tile pass, and with numeric columns
        # the long-field pass
        launches_per_step = 4 + (1 if any(t in ("i8", "i32", "i64", "f64") for t in w["cols"]) else 0)
    else:
        desc = pp.desc_json_lexer()
        T = info["n_tokens"]
        ids = torch.empty(T, dtype=torch.uint8, device=dev)
        starts = torch.empty(T, dtype=torch.int64, device=dev)
        lens = torch.empty(T, dtype=torch.int32, device=dev)
        status = pp.new_status(dev)

        def step():
            pp.pp_tokenize(d_in, n, desc, ids, starts, lens, T, status, stream)
        launches_per_step = 6  # init, stv, state scan, count, count scan, emit

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # correctness of the measured run: status must be clean and complete
    if csv:
        st = pp.read_status(out.status, len(w["cols"]))
        assert st["error"] == 0 and st["n_records"] == info["n_records"], st
        out_bytes = out.output_bytes(st["n_records"], st["chars_len"])
    else:
        st = pp.read_status(status)
        assert st["error"] == 0 and st["n_tokens"] == info["n_tokens"], st
        out_bytes = 13 * st["n_tokens"]

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    # per-kernel CUDA events of every timed call, on the launching stream
    pp.debug_stage_timing(args.steps)
    with Clocks(clock_index) as clk:
        _barrier(ws)
        torch.cuda.synchronize()
        t_start = time.perf_counter()
        for i in range(args.steps):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        _barrier(ws)
        wall = time.perf_counter() - t_start
    step_ms = [a.elapsed_time(b) for a, b in ev]
    tot_ms = _max_over_ranks(sum(step_ms), ws, dev)
    ms_per_step = tot_ms / args.steps
    value = n * ws * args.steps / (tot_ms / 1e3) / 1e9
    peak, peak_src = _peaks()
    path_s = float(np.mean(step_ms)) / 1e3
    st_ms = pp.debug_stage_ms(args.steps)
    pp.debug_stage_timing(0)
    names = (["init", "tile_stv_kernel", "tile_state_kernel", "parse_kernel", "long_field_kernel",
              "-"] if csv else
             ["init", "tok_stv_kernel", "tok_state_scan_kernel", "tok_count_kernel",
              "tok_count_scan_kernel", "tok_emit_kernel"])
    stages = {k: float(st_ms[:, i].mean()) for i, k in enumerate(names) if k != "-"}
    kernel = "parse_kernel" if csv else "tok_emit_kernel"
    kern_s = stages[kernel] / 1e3
    # the dominant kernel reads the input once and writes every output
    achieved = (n + out_bytes) / kern_s / 1e9

    # end to end through the public API with host buffers
    # the host link is shared with the machine's other jobs and its timings
    # vary from step to step: report the median of up to 5 steps
    e2e_steps = 0 if args.no_e2e else max(1, min(args.steps, 5))
    e2e_t = []
    h2d = d2h = 0
    if e2e_steps:  # pinned host outputs, allocated once like the device ones
        host_out = (pp.CsvOutputs(w["cols"], R, chars_cap, device="cpu") if csv
                    else pp.TokenOutputs(T))
    for i in range(e2e_steps + 1 if e2e_steps else 0):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        if csv:
            host_out.run_host(h_in, n, desc, stream=stream)
            est = pp.read_status(host_out.status, len(w["cols"]))
            h2d = n
            d2h = host_out.output_bytes(est["n_records"], est["chars_len"]) + pp.STATUS_BYTES
        else:
            est = host_out.run_host(h_in, n, desc, stream=stream)
            h2d = n
            d2h = 13 * est["n_tokens"] + pp.STATUS_BYTES
        dt = time.perf_counter() - t0
        assert est["error"] == 0, est
        if i > 0:
            e2e_t.append(dt)
    e2e_value = (n * ws / _max_over_ranks(float(np.median(e2e_t)), ws, dev) / 1e9) if e2e_t else None

    cpu = None
    if _dist()[1] == 0 and not args.no_cpu_baseline:
        cpu = _cpu_baseline(workload, h_in, info)
    traffic = _traffic(workload)
    rec = {
        "value": value, "ms_per_step": ms_per_step,
        "config": {"workload": workload, "n_bytes": n,
                   "n_records": info["n_records"] if csv else None,
                   "n_tokens": info["n_tokens"] if not csv else None,
                   "columns": w["cols"], "output_bytes": out_bytes,
                   "l2": "input (and output) larger than the 129 MB L2; no flush",
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "input_offset": off},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": n + out_bytes,
                     "kernel": kernel,
                     "timing": "CUDA events around the kernel on the launching stream, "
                               "every timed step"},
        "path": {"achieved_gbs": (n + out_bytes) / path_s / 1e9,
                 "frac": (n + out_bytes) / path_s / 1e9 / peak,
                 "kernel_ms": stages,
                 "note": "whole call (all kernels) against the same algorithmic bytes"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "timing": "median of %d steps after one warm-up, wall clock" % len(e2e_t),
                "api": "CsvOutputs.run_host (pp_parse_host: chunked host->device, parse, "
                       "device->host overlap) into pinned host outputs" if csv else
                       "TokenOutputs.run_host (pp_tokenize_host: chunked host->device, lexing, "
                       "device->host overlap) into pinned host triples"},
        "clocks": clk.summary(),
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_region": wall,
        "step_ms_min": min(step_ms), "step_ms_median": float(np.median(step_ms)),
    }
    del d_in, h_in
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import dfa_parsing_delimiter_gb300 as pp
    ws, rank, local = _dist()
    if ws > 1:
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    head = measure(pp, args.workload, args, dev, ws, local)
    # the other 2 GiB workload of the metric (the token stream lexed with the
    # 16-state DFA), reported beside the headline in the same line
    others = []
    if not args.no_others and args.target is None:
        other = "json_2gib" if args.workload != "json_2gib" else "csv18_2gib"
        others.append(measure(pp, other, args, dev, ws, local))
    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": head["value"], "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded generator, see datagen)",
    }
    line.update({k: v for k, v in head.items() if k not in ("value", "ms_per_step")})
    line["config"]["others"] = [
        dict({"metric": METRIC, "unit": "GB/s", "value": o["value"],
              "ms_per_step": o["ms_per_step"]},
             **{k: v for k, v in o.items() if k not in ("value", "ms_per_step")})
        for o in others]
    line["gpu_launches"] = head["gpu_launches"]
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(datagen.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--target", type=int, default=None,
                    help="input byte target (default: the workload's size); smaller "
                         "values give the small case used for ncu captures")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--in-offset", type=int, default=0,
                    help="place the device input this many bytes past an aligned "
                         "allocation (0-15: times the unaligned-input path)")
    ap.add_argument("--no-others", action="store_true",
                    help="time the headline workload only (not the second 2 GiB workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
