"""Benchmark: byte-level BPE encode throughput on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload serving|agentic]

One step = one tk_encode_segments call over the whole workload (split,
specials, safe chunking, merge, ordered assembly), inputs already in HBM.
Default workload: the serving batch (4,096 requests, 256 MiB; inputs larger
than L2, so no flush between steps). Prints one JSON line on rank 0.

--impl reference times the CPU oracle (the plain single-threaded encoder the
parity tests compare against) on a bounded sample of the same workload, on
this machine's host cores.
"""
import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BPE encode MB/s and tokens/s on 1 GB300 (IDs bit-exact), % of HBM roofline"


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
        desc = ("agentic prompt: ~4 M characters in 2,000 typed segments (alternating "
                "allow_special), prose/JSON/code/white-space runs up to 60k; tiktoken_safe=1")
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
    return table, np.ascontiguousarray(text), off, np.ascontiguousarray(allow), safe, desc


class Clocks:
    """nvidia-smi samples during the timed region."""

    def __init__(self, gpu_index):
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_{os.getpid()}.csv")
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
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
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
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
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    try:
        with open(os.path.join(root, "profiles", "traffic.txt")) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for name in ("tk_encode.cu", "tk_internal.cuh"):
            with open(os.path.join(root, "byte_level_bpe_gb300", "csrc", name), "rb") as f:
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


def run_gpu(args, rank, world):
    import torch

    import byte_level_bpe_gb300 as tk
    from byte_level_bpe_gb300 import native

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    table, text, off, allow, safe, desc = make_workload(args.workload, rank, args.total_mb)
    n, S = int(text.size), int(off.size - 1)
    tok = tk.Tokenizer(table, {k: v for k, v in __import__("workloads").SPECIALS.items()},
                       max_bytes=n, max_segments=S)
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
    native.tk_profile_enable(tok.workspace, True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(dev)
    if n > 160e6:
        # inputs larger than L2: back-to-back steps, one pair of events
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            n_ids = step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
    else:
        # inputs that fit in L2: flush it (write 256 MiB) before each step, outside
        # that step's events
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        evs = []
        for _ in range(args.steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            n_ids = step()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
        del flush
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    prof = native.tk_profile_read(tok.workspace)
    native.tk_profile_enable(tok.workspace, False)
    ms = max_over_ranks(ms, world)
    n_pt, _, n_long = native.tk_last_stats(tok.workspace)
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
        t0 = time.perf_counter()
        e2e_steps = max(1, min(args.steps, 5))
        for _ in range(e2e_steps):
            host_step()
        torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world)
    # warm word cache (reported apart from the cold headline): one call fills a
    # cross-call cache, then the same K steps are timed with it attached
    warm = None
    if not args.no_warm_cache:
        cache = native.tk_cache_create(tok.handle, max(n, 1 << 20))
        native.tk_workspace_set_cache(tok.workspace, cache)
        step()
        torch.cuda.synchronize()
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        for _ in range(args.steps):
            step()
        w1.record(stream)
        torch.cuda.synchronize()
        hits, _ = native.tk_last_cache_stats(tok.workspace)
        warm = {"ms_per_step": max_over_ranks(w0.elapsed_time(w1) / args.steps, world), "cache_hits": hits}
        native.tk_workspace_set_cache(tok.workspace, None)
        native.tk_cache_free(cache)
    return dict(n=n, S=S, n_ids=n_ids, n_pt=n_pt, n_long=n_long, ms=ms, e2e_ms=e2e_ms, prof=prof, clocks=clk,
                desc=desc, safe=safe, off=off, text=text, table=table, allow=allow, warm=warm)


def oracle_sample_rate(table, text, off, allow, safe, seconds=12.0):
    """Times the oracle on consecutive segments until ~`seconds` of CPU work."""
    import oracle
    import workloads
    enc = oracle.Encoding(table, workloads.SPECIALS)
    done_b, done_ids, t_used, s = 0, 0, 0.0, 0
    S = len(off) - 1
    while t_used < seconds and s < S:
        e = s
        while e < S and off[e] - off[s] < 2 << 20:
            e += 1
        e = max(e, s + 1)
        sub_text = text[off[s]:off[e]]
        sub_off = off[s:e + 1] - off[s]
        sub_allow = allow[s:e] if allow.size else np.zeros(e - s, np.uint8)
        t0 = time.perf_counter()
        ids, _ = enc.encode_arrays(sub_text, sub_off, sub_allow, e - s, safe)
        t_used += time.perf_counter() - t0
        done_b += int(sub_off[-1])
        done_ids += len(ids)
        s = e
    return done_b / t_used / 1e6, done_ids / t_used, done_b, s, t_used


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="serving", choices=["serving", "agentic", "prose", "multilingual"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--total-mb", type=int, default=256,
                    help="serving batch size in MiB (256 = the benchmark workload; smaller for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    ap.add_argument("--no-warm-cache", action="store_true", help="skip the warm word-cache leg")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl" if args.impl == "gb300" else "gloo")

    if args.impl == "reference":
        if rank != 0:
            return
        table, text, off, allow, safe, desc = make_workload(args.workload, 0, args.total_mb)
        for _ in range(max(0, min(args.warmup, 1))):
            pass
        rates = []
        for _ in range(args.steps):
            mbs, tps, nb, nseg, secs = oracle_sample_rate(table, text, off, allow, safe,
                                                          seconds=args.cpu_seconds / max(1, args.steps))
            rates.append((mbs, tps, nb, nseg, secs))
        mbs = float(np.median([r[0] for r in rates]))
        tps = float(np.median([r[1] for r in rates]))
        sample = f"first {rates[0][3]} segments ({rates[0][2]} bytes) per step, single thread"
        line = {"impl": "reference", "metric": METRIC, "value": round(mbs, 3), "unit": "MB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1e3 * float(np.median([r[4] for r in rates])), 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
                "data": "synthetic", "config": {"workload": desc, "impl_note": "CPU oracle"},
                "tokens_per_s": round(tps, 1),
                "cpu_baseline": {"value": round(mbs, 3), "unit": "MB/s", "cores": 1,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": round(mbs, 3), "unit": "MB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    r = run_gpu(args, rank, world)
    n, S, n_ids, n_pt, ms = r["n"], r["S"], r["n_ids"], r["n_pt"], r["ms"]
    peak, peak_kind = _peaks()
    total_n = n * world
    value = total_n / (ms * 1e-3) / 1e6
    tokens_per_s = n_ids * world / (ms * 1e-3)
    path_bytes = n + 4 * n_ids + 17 * S
    # dominant kernel of the timed region
    prof = r["prof"]
    steps = args.steps
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
                "algorithmic_bytes": int(kb)}
    launches = int(sum(v[1] for v in prof.values()))
    if rank != 0:
        return
    cpu_mbs = cpu_tps = cpu_s = float("nan")
    cpu_b = cpu_seg = 0
    if not args.no_cpu_baseline:
        cpu_mbs, cpu_tps, cpu_b, cpu_seg, cpu_s = oracle_sample_rate(
            r["table"], r["text"], r["off"], r["allow"], r["safe"], seconds=args.cpu_seconds)
    e2e_val = total_n / (r["e2e_ms"] * 1e-3) / 1e6
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "MB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic",
        "config": {"workload": r["desc"], "bytes": n, "segments": S, "pretokens": n_pt,
                   "ids": n_ids, "long_pretokens": r["n_long"], "l2": (f"inputs ({n / 2**20:.0f} MiB) larger than L2 (129 MB); no flush" if n > 160e6
                          else f"inputs ({n / 2**20:.1f} MiB) fit in L2 (129 MB): 256 MiB written "
                               "before each timed step, outside its events"),
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(tokens_per_s, 1),
        "path_roofline": {"bound": "hbm", "algorithmic_bytes": int(path_bytes),
                          "achieved": round(path_bytes / (ms * 1e-3) / 1e9, 1), "peak": peak,
                          "unit": "GB/s", "frac": round(path_bytes / (ms * 1e-3) / 1e9 / peak, 4)},
        "roofline": roof,
        "kernels_ms_per_step": {k: round(v[0] / steps, 4) for k, v in sorted(prof.items())},
        "cpu_baseline": {"value": round(cpu_mbs, 3), "unit": "MB/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {cpu_seg} requests ({cpu_b} bytes), single thread, "
                                   f"{cpu_s:.1f} s", "tokens_per_s": round(cpu_tps, 1)},
        "e2e": {"value": round(e2e_val, 2), "unit": "MB/s",
                "h2d_bytes_per_step": int(n + 8 * (S + 1) + S),
                "d2h_bytes_per_step": int(4 * n_ids + 8 * (S + 1) + 64)},
        "gpu_launches": launches,
        "warm_cache": None if r["warm"] is None else {
            "value": round(total_n / (r["warm"]["ms_per_step"] * 1e-3) / 1e6, 2), "unit": "MB/s",
            "ms_per_step": round(r["warm"]["ms_per_step"], 4), "cache_hits": r["warm"]["cache_hits"],
            "note": "cross-call word cache filled by one earlier call; the headline value is cold"},
        "clocks": r["clocks"],
    }
    print(json.dumps(_finite(line)))


def _finite(x):
    """NaN (a skipped leg) -> null, recursively."""
    if isinstance(x, dict):
        return {k: _finite(v) for k, v in x.items()}
    if isinstance(x, float) and x != x:
        return None
    return x


if __name__ == "__main__":
    main()
