"""Benchmark: byte-level BPE encode throughput on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload serving|agentic|multilingual|prose] [--no-sub]

One step = one tk_encode_segments call over the whole workload (split,
specials, safe chunking, merge, ordered assembly), inputs already in HBM.
Default workload: the serving batch (4,096 requests, 256 MiB; inputs larger
than L2, so no flush between steps). The headline is timed with the library's
per-kernel profiling off, one CUDA-event pair per step (median, p10, p90 and
mean reported); per-kernel times come from a second, profiled pass of the same
K steps. The million-token agentic prompt and the multilingual text are timed
the same way and reported as keyed sub-records of the same JSON line
("workloads"), each with its own roofline, CPU baseline and end-to-end figure.
Prints one JSON line on rank 0.

The CPU baseline is the oracle (the plain single-threaded encoder the parity
tests compare against) on one stated sample of each workload, in a child
process pinned to one host core, best of 3; its ids are compared with the
GPU's ids for the same segments ("ids_match"; a mismatch exits non-zero).
--impl reference times the same oracle on the same sample (the reference arm:
there is no reference code to install, the pages hold only prose).
"""
import argparse
import hashlib
import json
import multiprocessing as mp
import os
import platform
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BPE encode MB/s and tokens/s on 1 GB300 (IDs bit-exact), % of HBM roofline"

# Bytes of the oracle's sample per workload (about 10-30 s of single-core work
# for three timed runs at the oracle's ~4 MB/s).
CPU_SAMPLE_BYTES = 12 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def make_workload(name, rank=0, total_mb=256):
    import workloads
    table = workloads.full_table()
    if name == "serving":
        text, off = workloads.serving_batch(table, seed=5 + 1000 * rank, total=total_mb << 20,
                                            n_req=max(16, 4096 * total_mb // 256))
        allow = np.zeros(len(off) - 1, np.uint8)
        desc = (f"serving batch: {len(off) - 1:,} requests, log-normal lengths (median 8,192, "
                f"max 400,000), {total_mb} MiB total, 90% of each request repeats an earlier one; "
                "100,256-rank synthetic cl100k-shaped table; allow_special=0, tiktoken_safe=0")
        safe = False
    elif name == "agentic":
        segs = workloads.agentic_segments(table, seed=3 + 1000 * rank)
        text, off, allow = workloads.pack_segments(segs)
        desc = ("million-token agentic prompt: ~4 M characters in 2,000 typed segments "
                "(alternating allow_special), prose/JSON/code/white-space runs up to 60k; "
                "tiktoken_safe=1")
        safe = True
    elif name == "prose":
        text = np.frombuffer(workloads.prose_text(table, 1 << 20, seed=2 + 1000 * rank), np.uint8)
        off = np.array([0, text.size], np.int64)
        allow = np.zeros(1, np.uint8)
        desc = ("full-size table, 1 MiB of mixed text (Zipf over the table's letter tokens with "
                "punctuation, digits and newlines), one segment, tiktoken_safe=0")
        safe = False
    elif name == "multilingual":
        ext = workloads.multilingual_table(table)
        table = [(t, i) for i, t in enumerate(table)] + ext
        text = workloads.multilingual_text(workloads.full_table(), seed=4 + 1000 * rank)
        text = np.frombuffer(text.tobytes() if isinstance(text, np.ndarray) else bytes(text), np.uint8)
        off = np.array([0, text.size], np.int64)
        allow = np.zeros(1, np.uint8)
        desc = ("multilingual UTF-8 stress: table + 20,000 merges over UTF-8 byte sequences, 8 MiB "
                "(ASCII 35%, CJK 30%, Devanagari 20%, emoji 10%, control bytes 5%), one segment")
        safe = False
    else:
        raise SystemExit(f"unknown workload {name}")
    return table, np.ascontiguousarray(text), np.ascontiguousarray(off, np.int64), \
        np.ascontiguousarray(allow), safe, desc


def input_sha256(text, off, allow):
    import workloads
    return workloads.input_sha256(text, off, allow)


class Clocks:
    """nvidia-smi samples during the timed region (written to a temporary file)."""

    def __init__(self, gpu_index):
        self.proc = None
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.seek(0)
        lines = self.f.read().splitlines()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


# Algorithmic HBM bytes of each kernel per launch (stated in the design notes):
# n = input bytes, p = pre-tokens, t = ids, s = segments.
def kernel_bytes(name, n, p, t, s):
    return {
        # read the text and the segment table, write the pre-token start bitmap
        "k_split": n + n // 8 + 8 * (s + 1),
        # read the text and the start bitmap, write the ids and the segment offsets
        "k_encode_tiles": n + n // 8 + 4 * t + 16 * (s + 1),
        "k_chunk_scan_windows": n + n // 8,
        "k_chunk_scan_runs": n + n // 8,
    }.get(name)


def captured_traffic(kernel, n):
    """DRAM bytes per launch of `kernel` from the committed ncu capture
    (profiles/traffic.txt), scaled to n input bytes; None when the kernel
    sources changed after the capture or the kernel was not captured."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.txt")) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for name in ("tk_encode.cu", "tk_internal.cuh"):
            with open(os.path.join(ROOT, "byte_level_bpe_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
    except (OSError, ValueError):
        return None
    k = rec.get("kernels", {}).get(kernel)
    if h.hexdigest()[:16] != rec.get("source_sha256_prefix") or not k:
        return None
    return int(k["dram_bytes"] * n / k["input_bytes"])


def max_over_ranks(x, world, device="cuda"):
    """The largest x over the ranks (x itself on one rank): the job's time is
    its slowest replica's."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU leg: the oracle in a child process pinned to one host core.

def host_cpu():
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"model": model or platform.processor() or platform.machine(),
            "arch": platform.machine(), "nproc": os.cpu_count()}


def cpu_sample(off, budget=CPU_SAMPLE_BYTES):
    """The oracle's sample: the workload's first segments, up to `budget` bytes
    (at least one segment; a segment longer than the budget is taken whole)."""
    S = len(off) - 1
    e = 1
    while e < S and off[e + 1] <= budget:
        e += 1
    return 0, e


def _oracle_child(table, text, off, allow, safe, warmup, runs, core):
    """Runs in a spawned process: pins itself to `core`, builds the oracle's
    tables (untimed), encodes the sample `warmup` times untimed, then `runs`
    timed times; returns the wall times and the ids of the last run."""
    try:
        os.sched_setaffinity(0, {core})
        pinned = sorted(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        pinned = None
    import oracle
    import workloads
    enc = oracle.Encoding(table, workloads.SPECIALS)
    S = len(off) - 1
    for _ in range(warmup):
        enc.encode_arrays(text, off, allow, S, safe)
    times, ids = [], None
    for _ in range(runs):
        t0 = time.perf_counter()
        ids, offs = enc.encode_arrays(text, off, allow, S, safe)
        times.append(time.perf_counter() - t0)
    return times, ids, offs, pinned


def oracle_leg(table, text, off, allow, safe, warmup=1, runs=3):
    s, e = cpu_sample(off)
    sub_text = np.ascontiguousarray(text[off[s]:off[e]])
    sub_off = np.ascontiguousarray(off[s:e + 1] - off[s])
    sub_allow = np.ascontiguousarray(allow[s:e] if allow.size >= e else np.zeros(e - s, np.uint8))
    core = max(0, (os.cpu_count() or 1) - 1)
    ctx = mp.get_context("spawn")
    with ctx.Pool(1) as pool:
        times, ids, offs, pinned = pool.apply(_oracle_child, (table, sub_text, sub_off, sub_allow, safe,
                                                              warmup, runs, core))
    nb = int(sub_off[-1])
    return {"times": times, "ids": ids, "offs": offs, "bytes": nb, "segments": (s, e), "core": core,
            "pinned": pinned}


def cpu_record(leg, cpu):
    best = min(leg["times"])
    return {"value": round(leg["bytes"] / best / 1e6, 3), "unit": "MB/s", "cores": 1, "kind": "oracle",
            "tokens_per_s": round(len(leg["ids"]) / best, 1),
            "sample": (f"segments {leg['segments'][0]}..{leg['segments'][1] - 1} "
                       f"({leg['bytes']:,} bytes, {len(leg['ids']):,} ids): the workload's first segments "
                       f"up to {CPU_SAMPLE_BYTES >> 20} MiB; best of {len(leg['times'])} runs after "
                       f"1 untimed run, single thread pinned to core {leg['core']}"),
            "runs_s": [round(t, 3) for t in leg["times"]],
            "pinned_cores": leg["pinned"], "host_cpu": cpu}


# ---------------------------------------------------------------------------
# GPU leg.

def time_steps(step, steps, stream, flush):
    """K steps, one CUDA-event pair each on the launching stream; with `flush`
    (inputs that fit in L2) 256 MiB is written before each step, outside its
    events. Returns the per-step milliseconds."""
    import torch
    evs = []
    for _ in range(steps):
        if flush is not None:
            flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def run_gpu(name, args, rank, world, headline):
    import torch

    import byte_level_bpe_gb300 as tk
    import workloads
    from byte_level_bpe_gb300 import native

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    table, text, off, allow, safe, desc = make_workload(name, rank, args.total_mb if name == "serving" else 256)
    n, S = int(text.size), int(off.size - 1)
    tok = tk.Tokenizer(table, dict(workloads.SPECIALS), max_bytes=n, max_segments=S)
    d_text = torch.from_numpy(text).cuda()
    d_off = torch.from_numpy(off).cuda()
    d_allow = torch.from_numpy(allow if allow.size else np.zeros(1, np.uint8)).cuda()
    out = torch.empty(n, dtype=torch.int32, device="cuda")
    out_off = torch.empty(S + 1, dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        return native.tk_encode_segments(tok.handle, tok.workspace, d_text.data_ptr(), n,
                                         d_off.data_ptr(), d_allow.data_ptr(), S, safe,
                                         out.data_ptr(), n, out_off.data_ptr(), stream.cuda_stream)[1]

    for _ in range(args.warmup):
        n_ids = step()
    flush = None if n > 160e6 else torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    # headline: profiling off
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(dev) if headline else None
    step_ms = time_steps(step, args.steps, stream, flush)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    n_pt, n_ids, n_long = native.tk_last_stats(tok.workspace)
    ids_dev, off_dev = out[:n_ids].cpu().numpy(), out_off.cpu().numpy()
    # per-kernel times: a second pass of K steps with the library's events on
    native.tk_profile_enable(tok.workspace, True)
    prof_ms = time_steps(step, args.steps, stream, flush)
    prof = native.tk_profile_read(tok.workspace)
    native.tk_profile_enable(tok.workspace, False)
    # e2e: host buffers through tk_encode_segments_host (H2D + encode + D2H each step)
    h_text = torch.from_numpy(text).pin_memory().numpy()
    h_off = torch.from_numpy(off).pin_memory().numpy()
    h_allow = torch.from_numpy(allow if allow.size else np.zeros(1, np.uint8)).pin_memory().numpy()
    h_out = torch.empty(n, dtype=torch.int32).pin_memory().numpy()
    h_out_off = torch.empty(S + 1, dtype=torch.int64).pin_memory().numpy()

    def host_step():
        return native.tk_encode_segments_host(tok.handle, tok.workspace, h_text.ctypes.data, n,
                                              h_off.ctypes.data, h_allow.ctypes.data, S, safe,
                                              h_out.ctypes.data, n, h_out_off.ctypes.data,
                                              stream.cuda_stream)[1]

    e2e_ms = float("nan")
    if not args.no_e2e:
        host_step()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e2e_steps = max(1, min(args.steps, 5))
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            host_step()
        torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
        assert np.array_equal(h_out[:n_ids], ids_dev), "host-buffer call differs from the device call"
    warm = None
    if headline and not args.no_warm_cache:
        # warm word cache (reported apart from the cold headline): one call fills a
        # cross-call cache, then the same K steps are timed with it attached
        cache = native.tk_cache_create(tok.handle, max(n, 1 << 20))
        native.tk_workspace_set_cache(tok.workspace, cache)
        step()
        warm_ms = time_steps(step, args.steps, stream, flush)
        hits, _ = native.tk_last_cache_stats(tok.workspace)
        warm = {"ms_per_step": max_over_ranks(float(np.mean(warm_ms)), world), "cache_hits": hits}
        native.tk_workspace_set_cache(tok.workspace, None)
        native.tk_cache_free(cache)
    tok.close()
    del d_text, out, flush
    torch.cuda.empty_cache()
    return dict(name=name, n=n, S=S, n_ids=n_ids, n_pt=n_pt, n_long=n_long, step_ms=step_ms,
                prof_ms=prof_ms, e2e_ms=max_over_ranks(e2e_ms, world), prof=prof, clocks=clk,
                desc=desc, safe=safe, off=off, text=text, table=table, allow=allow, warm=warm,
                ids=ids_dev, g_off=off_dev, sha=input_sha256(text, off, allow))


def manifest_entry(name, total_mb, rank=0):
    """The recorded sha256 of a workload input (workloads/manifest.json), or
    None (a serving batch of another size, another rank's seed, or prose)."""
    try:
        with open(os.path.join(ROOT, "workloads", "manifest.json")) as f:
            m = json.load(f)
    except (OSError, ValueError):
        return None
    if rank != 0 or (name == "serving" and total_mb != 256):
        return None
    return m.get("inputs", {}).get(name, {}).get("sha256")


def record(r, args, world, cpu, peak, peak_kind):
    """The JSON record of one workload (headline fields + roofline + baselines)."""
    n, S, n_ids, n_pt = r["n"], r["S"], r["n_ids"], r["n_pt"]
    steps = args.steps
    ms_steps = [max_over_ranks(x, world) for x in r["step_ms"]]
    ms = float(np.mean(ms_steps))
    total_n = n * world
    path_bytes = n + 4 * n_ids + 17 * S
    prof = r["prof"]
    dom = max((k for k in prof if kernel_bytes(k, n, n_pt, n_ids, S) is not None),
              key=lambda k: prof[k][0], default=None)
    roof = None
    if dom:
        avg_ms = prof[dom][0] / prof[dom][1]
        kb = kernel_bytes(dom, n, n_pt, n_ids, S)
        ach = kb / (avg_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": round(ach, 1), "peak": peak,
                "unit": "GB/s", "frac": round(ach / peak, 4), "traffic": captured_traffic(dom, n),
                "peak_source": peak_kind, "kernel_ms": round(avg_ms, 4),
                "algorithmic_bytes": int(kb),
                "timing": "CUDA events on each kernel's own stream, in a profiled pass of the same "
                          "K steps right after the headline pass"}
    launches_per_step = int(sum(v[1] for v in prof.values())) / max(1, steps)
    leg = None if args.no_cpu_baseline else oracle_leg(r["table"], r["text"], r["off"], r["allow"], r["safe"])
    ids_match = None
    if leg is not None:
        s, e = leg["segments"]
        got = r["ids"][r["g_off"][s]:r["g_off"][e]]
        ids_match = bool(np.array_equal(got, leg["ids"]) and
                         np.array_equal(r["g_off"][s:e + 1] - r["g_off"][s], leg["offs"]))
    exp_sha = manifest_entry(r["name"], args.total_mb)
    e2e_val = total_n / (r["e2e_ms"] * 1e-3) / 1e6
    line = {
        "metric": METRIC, "value": round(total_n / (ms * 1e-3) / 1e6, 2), "unit": "MB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "step_ms": {"median": round(float(np.median(ms_steps)), 4),
                    "p10": round(float(np.percentile(ms_steps, 10)), 4),
                    "p90": round(float(np.percentile(ms_steps, 90)), 4),
                    "mean": round(ms, 4), "timing": "one CUDA-event pair per step on the launching "
                                                     "stream, library profiling off; max over ranks"},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic",
        "config": {"workload": r["desc"], "bytes": n, "segments": S, "pretokens": n_pt,
                   "ids": n_ids, "long_pretokens": r["n_long"],
                   "input_sha256": r["sha"], "manifest_sha256_match": (None if exp_sha is None
                                                                       else exp_sha == r["sha"]),
                   "l2": (f"inputs ({n / 2**20:.0f} MiB) larger than L2 (129 MB); no flush" if n > 160e6
                          else f"inputs ({n / 2**20:.1f} MiB) fit in L2 (129 MB): 256 MiB written "
                               "before each timed step, outside its events"),
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(n_ids * world / (ms * 1e-3), 1),
        "path_roofline": {"bound": "hbm", "algorithmic_bytes": int(path_bytes),
                          "achieved": round(path_bytes / (ms * 1e-3) / 1e9, 1), "peak": peak,
                          "unit": "GB/s", "frac": round(path_bytes / (ms * 1e-3) / 1e9 / peak, 4),
                          "peak_source": peak_kind},
        "roofline": roof,
        "kernels_ms_per_step": {k: round(v[0] / steps, 4) for k, v in sorted(prof.items())},
        "profiled_ms_per_step": round(float(np.mean(r["prof_ms"])), 4),
        "cpu_baseline": None if leg is None else cpu_record(leg, cpu),
        "ids_match": ids_match,
        "e2e": {"value": round(e2e_val, 2), "unit": "MB/s",
                "h2d_bytes_per_step": int(n + 8 * (S + 1) + S),
                "d2h_bytes_per_step": int(4 * n_ids + 8 * (S + 1) + 64)},
        "gpu_launches": int(round(launches_per_step * steps)),
    }
    if r["warm"] is not None:
        line["warm_cache"] = {
            "value": round(total_n / (r["warm"]["ms_per_step"] * 1e-3) / 1e6, 2), "unit": "MB/s",
            "ms_per_step": round(r["warm"]["ms_per_step"], 4), "cache_hits": r["warm"]["cache_hits"],
            "note": "cross-call word cache filled by one earlier call; the headline value is cold"}
    if r["clocks"] is not None:
        line["clocks"] = r["clocks"]
    return line


def reference_arm(args, rank):
    """The oracle alone on the same stated sample as the GPU arm's CPU baseline:
    W untimed runs, then K timed runs in a child pinned to one core."""
    if rank != 0:
        return
    table, text, off, allow, safe, desc = make_workload(args.workload, 0, args.total_mb)
    leg = oracle_leg(table, text, off, allow, safe, warmup=args.warmup, runs=args.steps)
    rates = [leg["bytes"] / t / 1e6 for t in leg["times"]]
    mbs = float(np.median(rates))
    rec = cpu_record(leg, host_cpu())
    rec["value"] = round(mbs, 3)
    rec["sample"] = rec["sample"].replace(f"best of {len(leg['times'])} runs after 1 untimed run",
                                          f"median of {len(leg['times'])} runs after {args.warmup} "
                                          "untimed runs")
    line = {"impl": "reference", "metric": METRIC, "value": round(mbs, 3), "unit": "MB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * float(np.median(leg["times"])), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic",
            "config": {"workload": desc, "impl_note": "CPU oracle on the stated sample of the workload",
                       "input_sha256": input_sha256(text, off, allow)},
            "tokens_per_s": round(len(leg["ids"]) / float(np.median(leg["times"])), 1),
            "cpu_baseline": rec,
            "e2e": {"value": round(mbs, 3), "unit": "MB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="serving", choices=["serving", "agentic", "prose", "multilingual"])
    ap.add_argument("--total-mb", type=int, default=256,
                    help="serving batch size in MiB (256 = the benchmark workload; smaller for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing legs")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer legs")
    ap.add_argument("--no-warm-cache", action="store_true", help="skip the warm word-cache leg")
    ap.add_argument("--no-sub", action="store_true",
                    help="skip the agentic and multilingual sub-records")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        raise SystemExit("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl" if args.impl == "gb300" else "gloo")

    if args.impl == "reference":
        reference_arm(args, rank)
        return

    peak, peak_kind = _peaks()
    cpu = host_cpu()
    r = run_gpu(args.workload, args, rank, world, headline=True)
    subs = []
    if not args.no_sub and args.workload == "serving":
        subs = [run_gpu(w, args, rank, world, headline=False) for w in ("agentic", "multilingual")]
    if rank != 0:
        return
    line = record(r, args, world, cpu, peak, peak_kind)
    if subs:
        line["workloads"] = {s["name"]: record(s, args, world, cpu, peak, peak_kind) for s in subs}
    print(json.dumps(_finite(line)))
    bad = [k for k, v in [(args.workload, line)] + list(line.get("workloads", {}).items())
           if v.get("ids_match") is False]
    if bad:
        print(f"ids differ from the oracle on the sample of: {', '.join(bad)}", file=sys.stderr)
        sys.exit(1)


def _finite(x):
    """NaN (a skipped leg) -> null, recursively."""
    if isinstance(x, dict):
        return {k: _finite(v) for k, v in x.items()}
    if isinstance(x, list):
        return [_finite(v) for v in x]
    if isinstance(x, float) and x != x:
        return None
    return x


if __name__ == "__main__":
    main()
