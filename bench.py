"""Benchmark of the paged KV cache hot path on GB300.

One step = one pass of the whole path over one batch of the Llama-3-8B-shaped
decode workload (32 requests, contexts uniform in [512, 4096], H_q 32,
H_kv 8, head_dim 128, block_size 64, bf16): manager->kernel block
expansion, slot mapping of the step's tokens and the K/V cache scatter (one
fused kernel), and the paged decode (partition + merge kernels).  Inputs
are seeded, synthetic and resident in HBM; the caches were filled
beforehand through the same library.  L2 is flushed (a write of 2x the L2
size, read back) before every timed step, outside the timed interval.

value  = decode KV bytes needed per step (cache_len rows x K,V x H_kv x D x 2B)
         / device time of the step (CUDA events), aggregated over ranks.
e2e    = the same bytes / time of a step that also copies the step's inputs
         from pinned host memory and reads the output back.
roofline.achieved = the same bytes / device time of the decode partition
         kernel alone (the dominant kernel; bkv_paged_decode_partition);
         decode_ms is the whole decode call (partition + merge).
secondary = slot mapping + cache write of the ragged mixed step (tokens/s).

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl bkv|reference]
                  [--workload NAME] [--sliding-window W] [--kv-dtype bf16|fp8]
                  [--cp-world W [--cp-interleave I]] [--attention decode|ragged]
                  [--part step|write] [--eager] [--no-cpu-baseline] [--no-secondary]
--workload / --sliding-window / --kv-dtype / --cp-world time another seeded
workload, a sliding-window decode, FP8 caches or one decode-context-parallel
rank on the same harness; --attention ragged times the mixed-step attention
(tensor roofline); --part write times slot mapping + cache write of the
ragged step alone.  The default is the headline configuration above.
Under torchrun every rank runs an independent replica (the path has no
exchange step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-decode KV-read GB/s (% HBM peak); slot-map+cache-write tokens/s"
WORKLOAD = "llama3_decode"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "paged_decode_llama3_decode.txt")
DECODE_SOURCES = ["bkv_decode.cu", "bkv_decode_tc.cu", "bkv_decode.cuh"]


# per-tensor scales of the FP8 runs: the Llama-shaped K/V draws (sd 1/sqrt(128)) span about +-0.4,
# well inside 448 * scale
FP8_SCALES = (2.0 ** -9, 1e-3)


def _dist():
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl")
        return dist
    return None


def max_over_ranks(values, dist, device="cpu"):
    """Each value's maximum over the ranks of the job (the values themselves at one rank): a step
    time is that of the slowest replica."""
    if not dist:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _describe(w, window, cp=(1, 0, 1), fp8=None):
    """The workload's name and sizes, as the JSON line's config.workload."""
    if fp8 is not None:
        return (_describe(w, window, cp) + f", E4M3 KV cache (k_scale {fp8[0]:g}, v_scale {fp8[1]:g}; 1 byte per "
                "element, K and V used as loaded by E4M3 tensor cores)")
    if cp[0] > 1:
        return (_describe(w, window) + f", decode-context-parallel rank {cp[1]} of {cp[0]} (interleave {cp[2]}): "
                f"its own share of every request's keys")
    if w.name == WORKLOAD and window == 0:
        return ("llama3_decode: 32 req, ctx U[512,4096] + 1 new token, H_q 32, H_kv 8, D 128, bs 64, bf16, "
                "fp32 accumulate")
    lens = w.context_lens[: w.num_real]
    bs = (f"bs {w.block_size} -> kernel bs {w.kernel_block_size}" if w.block_size != w.kernel_block_size
          else f"bs {w.block_size}")
    d = (f"{w.name}: {w.num_real} req" + (f" + {w.num_rows - w.num_real} NULL rows" if w.num_rows > w.num_real
                                          else "")
         + f", ctx {int(lens.min())}..{int(lens.max())} (mean {lens.mean():.0f}), q_len {w.q_len}, H_q "
         f"{w.num_q_heads}, H_kv {w.num_kv_heads}, D {w.head_dim}, {bs}, {w.dtype}, fp32 accumulate")
    return d + (f", sliding window {window}" if window else "")


def _code_only(text):
    """C/CUDA source without comments or blank lines, runs of blanks as one space (string literals in
    these sources hold neither comment markers nor blank runs), so that a comment edit does not count
    as a new kernel."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(" ".join(line.split()) for line in text.splitlines() if line.strip())


def _decode_source_sha():
    """Hash of the decode kernels' code (comments ignored): the committed ncu summary's traffic line
    is reported only while it matches."""
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        p = os.path.join(ROOT, "paged_kv_cache_slot_gb300", "csrc", f)
        if os.path.exists(p):
            h.update(_code_only(open(p).read()).encode())
    return h.hexdigest()[:16]


def _profiled_traffic():
    """dram bytes per decode launch from the committed ncu summary, if it still
    describes the current kernel source (else None)."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    kv = {}
    for line in open(PROFILE_TRAFFIC):
        if ":" in line:
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("decode_source_sha256") != _decode_source_sha():
        return None
    try:
        return int(kv["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the raw samples: BKV_CLOCKS_CSV if set (a path to keep them), else a temporary file
        self.path = os.environ.get("BKV_CLOCKS_CSV") or os.path.join(
            tempfile.gettempdir(), f"bkv_clocks_{os.getpid()}_{index}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        # the timed region lasts well under a second: start it only once the sampler is live
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 5.0 and self.proc.poll() is None:
            self.fh.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _oracle_pass(oracle, rows, q, kc, vc, table, ctx, window, threads):
    """The oracle's decode of ``rows`` (longest first), one request per call, on ``threads`` host threads
    (the C oracle runs with the interpreter lock released, so the calls run in parallel)."""
    if threads <= 1:
        for r in rows:
            oracle.paged_decode_request(r, q, kc, vc, table, ctx, sliding_window=window)
        return
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda r: oracle.paged_decode_request(r, q, kc, vc, table, ctx, sliding_window=window), rows))


def _cpu_baseline(budget_s: float, workload: str = WORKLOAD, window: int = 0):
    """The oracle, as it stands, on the whole workload: every request decoded (fp64), timed once over all
    host cores (threads over requests, longest first) and once on a single thread, each pass repeated
    until about ``budget_s`` / 2 of CPU work.  The all-cores figure is the baseline; the single-thread
    one is reported beside it."""
    import oracle
    from oracle.cases import fill_oracle_cache
    from paged_kv_cache_slot_gb300 import workloads as wl

    w = wl.make(workload)
    q = w.q()
    kc, vc, table = fill_oracle_cache(w)
    rows = [int(r) for r in np.argsort(w.context_lens, kind="stable")[::-1] if w.context_lens[r] > 0]
    per_tok = 2 * w.num_kv_heads * w.head_dim * w.elem_bytes
    Ls = w.context_lens.astype(np.int64)
    eff = Ls - (np.maximum(0, Ls - w.q_len - window + 1) if window > 0 else 0)   # rows each request reads
    pass_bytes = int(eff.sum()) * per_tok
    cores = os.cpu_count() or 1

    def timed(threads):
        t0 = time.perf_counter()
        _oracle_pass(oracle, rows, q, kc, vc, table, w.context_lens, window, threads)
        first = time.perf_counter() - t0
        reps = max(1, math.ceil((budget_s / 2) / max(first, 1e-6)) - 1)
        t0 = time.perf_counter()
        for _ in range(reps):
            _oracle_pass(oracle, rows, q, kc, vc, table, w.context_lens, window, threads)
        dt = time.perf_counter() - t0
        return pass_bytes * reps / dt / 1e9, reps, dt

    v_all, reps_all, t_all = timed(cores)
    v_one, reps_one, t_one = timed(1)
    model = cpu_model()
    return {"value": v_all, "unit": "GB/s", "cores": cores, "kind": "oracle", "cpu_model": model,
            "sample": f"all {len(rows)} requests of {workload} ({pass_bytes / 1e6:.1f} MB of K/V per pass) decoded by "
                      f"the fp64 C oracle, {reps_all} passes in {t_all:.1f} s on {cores} threads (requests in "
                      f"parallel, longest first)",
            "single_thread": {"value": v_one, "unit": "GB/s", "cores": 1,
                              "sample": f"{reps_one} passes in {t_one:.1f} s on one thread"}}


def run_reference(args):
    """--impl reference: the oracle, as it stands, on the host cores, with this arm's metric and config:
    each step is the whole headline step of the Llama-shaped batch -- block expansion, slot mapping and
    cache write of the step's 32 tokens, and the decode of all 32 requests (threads over requests on
    every core) -- over caches the oracle filled beforehand."""
    dist = _dist()
    rank = dist.get_rank() if dist else 0
    if rank != 0:
        return
    import oracle
    from oracle.cases import fill_oracle_cache
    from paged_kv_cache_slot_gb300 import workloads as wl

    w = wl.make(WORKLOAD)
    q = w.q()
    w_prior = wl.make(WORKLOAD)
    w_prior.new_tokens = np.zeros_like(w_prior.new_tokens)      # the caches before this step: prior tokens only
    kc, vc, _ = fill_oracle_cache(w_prior)
    req, pos = w.step_tokens()
    kn, vn = w.step_kv()
    per_tok = 2 * w.num_kv_heads * w.head_dim * w.elem_bytes
    step_bytes = int(w.context_lens.astype(np.int64).sum()) * per_tok
    rows = [int(r) for r in np.argsort(w.context_lens, kind="stable")[::-1]]
    cores = os.cpu_count() or 1

    def one_step():
        t0 = time.perf_counter()
        table = oracle.map_to_kernel_blocks(w.block_table, w.block_size, w.kernel_block_size)
        slots, _ = oracle.compute_slot_mapping(table, req, pos, w.kernel_block_size, w.num_tokens, w.max_num_tokens)
        oracle.cache_write(kn, vn, slots, kc, vc, num_tokens=w.num_tokens, inplace=True)
        _oracle_pass(oracle, rows, q, kc, vc, table, w.context_lens, 0, cores)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        one_step()
    times = [one_step() for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    value = step_bytes / (ms / 1e3) / 1e9
    sample = (f"the whole step per timed step: block expansion, slot mapping + cache write of 32 tokens and the "
              f"decode of all 32 requests ({step_bytes / 1e6:.1f} MB of K/V) by the fp64 C oracle on {cores} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": _describe(w, 0), "sample": "every request of the workload, every step"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bucket_report(w):
    """The long-context decode's K/V bytes three ways ("Decode Context-Length Bucketing", Problem: a
    request that reads its full max_model_len row of the block table moves far more than its context;
    Design / Per-step bucket selection: needed_seq = max(num_computed) + 1 + num_speculative_tokens and
    the bucket is the smallest configured length >= needed_seq, max_model_len last): what the decode
    reads (each request's cache_len rows), the full rows, and the chosen bucket's rows for every
    request of the batch."""
    per_tok = 2 * w.num_kv_heads * w.head_dim * w.elem_bytes
    spec = w.q_len - 1
    needed = int(w.prior_lens[: w.num_real].max()) + 1 + spec
    mml = int(w.extra["max_model_len"])
    cands = sorted(int(b) for b in w.extra["buckets"]) + [mml]
    bucket = next((b for b in cands if b >= needed), -1)
    read = int(w.context_lens[: w.num_real].astype(np.int64).sum()) * per_tok
    full = w.num_real * mml * per_tok
    bucketed = w.num_real * bucket * per_tok if bucket > 0 else None
    return {"workload": w.name, "needed_seq": needed, "buckets": cands, "bucket": bucket,
            "kv_bytes_read": read, "full_row_bytes": full, "bucketed_bytes": bucketed,
            "full_row_over_read": full / read, "bucketed_over_read": (bucketed / read) if bucketed else None,
            "source": "Decode Context-Length Bucketing: Problem (~32x DMA amplification of full-row reads, "
                      "Trn2/Trn3) and Design / Per-step bucket selection"}


def torch_int64():
    import torch
    return torch.int64


def _flush_l2(flush):
    """Evict L2 before a timed step: write a buffer of 2x the L2 size, then
    read it back, so that the dirty lines of the write are written back here
    and not during the timed step."""
    flush.zero_()
    flush.view(torch_int64()).amax()


def _time_steps(torch, fn, steps, flush, stream):
    """Per-step device times (ms) with an L2 flush before each step, outside the events."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            _flush_l2(flush)
            a.record(stream)
            fn()
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def run_bkv(args):
    import torch

    from paged_kv_cache_slot_gb300 import bkv
    from paged_kv_cache_slot_gb300 import workloads as wl
    from paged_kv_cache_slot_gb300.build import build
    from paged_kv_cache_slot_gb300.staging import DeviceWorkload

    dist = _dist()
    rank = dist.get_rank() if dist else 0
    world = dist.get_world_size() if dist else 1
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if rank == 0:
        build()
    if dist:
        dist.barrier()
    bkv.load()
    if args.decode_kernel == "generic":
        # the CUDA-core partition kernel on every shape (a comparison switch the library never sets)
        bkv.load().bkv_testing_force_generic_decode(1)

    w = wl.make(args.workload)
    cp = (args.cp_world, 0, args.cp_interleave)
    fp8 = FP8_SCALES if args.kv_dtype == "fp8" else None
    dw = DeviceWorkload(w, device=f"cuda:{local}", sliding_window=args.sliding_window, cp_world=cp[0],
                        cp_rank=cp[1], cp_interleave=cp[2], kv_fp8=fp8)
    headline = (args.workload == WORKLOAD and args.sliding_window == 0 and cp[0] == 1 and fp8 is None
                and args.decode_kernel == "auto")
    stream = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = torch.empty(2 * max(l2, 64 << 20), dtype=torch.uint8, device=f"cuda:{local}")
    kv_bytes = dw.decode_kv_bytes()

    def step():
        dw.step(stream=stream)

    def decode_only():
        dw.decode(stream=stream)

    def partition_only():
        if cp[0] > 1:      # no separate phases for a context-parallel rank: the whole decode call
            dw.decode(stream=stream)
        else:
            dw.decode_partition(stream=stream)

    # End-to-end leg: the step's inputs live packed in one pinned host buffer and one device
    # buffer (each tensor at a 256-byte aligned offset; the device tensors the library reads are
    # views of it), so a step uploads them with one host-to-device copy, as a serving engine that
    # stages its per-step inputs in one buffer would, and reads the output back with one copy.
    in_names = ("mgr_table", "req_indices", "positions", "k_new", "v_new", "q", "context_lens")
    spans, off = {}, 0
    for name in in_names:
        t = getattr(dw, name)
        spans[name] = (off, t.numel() * t.element_size())
        off = (off + spans[name][1] + 255) // 256 * 256
    dev_in = torch.zeros(off, dtype=torch.uint8, device=f"cuda:{local}")
    host_in = torch.zeros(off, dtype=torch.uint8, pin_memory=True)
    for name in in_names:
        t = getattr(dw, name)
        o, n = spans[name]
        host_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        view = dev_in[o:o + n].view(t.dtype).view(t.shape)
        view.copy_(t)
        setattr(dw, name, view)
    host_out = torch.empty(dw.out.shape, dtype=dw.out.dtype, pin_memory=True)
    h2d_bytes = off
    d2h_bytes = host_out.numel() * host_out.element_size()

    def e2e_step():
        dev_in.copy_(host_in, non_blocking=True)
        dw.step(stream=stream)
        host_out.copy_(dw.out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
            e2e_step()
            decode_only()
            partition_only()
    torch.cuda.synchronize()

    # CUDA graphs of the three timed bodies (a serving engine replays its
    # decode step as a graph); captured after the warm-up so that one-time
    # set-up (kernel attributes, driver entry points) is outside the graphs.
    BODIES = (("step", step), ("decode", decode_only), ("partition", partition_only), ("e2e", e2e_step))
    graphs = {}
    if not args.eager:
        for name, fn in BODIES:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            graphs[name] = g
        torch.cuda.synchronize()
        for g in graphs.values():
            g.replay()
        torch.cuda.synchronize()
    body = {name: (graphs[name].replay if name in graphs else fn)
            for name, fn in BODIES}

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        step_ms = _time_steps(torch, body["step"], args.steps, flush, stream)
        dec_ms = _time_steps(torch, body["decode"], args.steps, flush, stream)
        part_ms = _time_steps(torch, body["partition"], args.steps, flush, stream)
        e2e_ms = _time_steps(torch, body["e2e"], args.steps, flush, stream)
        t_wall = time.perf_counter() - t_wall0
    eager_ms = None
    if graphs:
        eager_ms = statistics.mean(_time_steps(torch, step, args.steps, flush, stream))
    torch.cuda.synchronize()
    if dist:
        dist.barrier()

    ms = sum(step_ms) / len(step_ms)
    dms = sum(dec_ms) / len(dec_ms)
    ems = sum(e2e_ms) / len(e2e_ms)
    pms = sum(part_ms) / len(part_ms)
    ms, dms, ems, pms = max_over_ranks([ms, dms, ems, pms], dist, f"cuda:{local}")

    # context parallelism: the merge of cp_world ranks' (out, lse) that follows their exchange
    cp_merge = None
    if rank == 0 and cp[0] > 1:
        outs = torch.stack([dw.out] * cp[0])
        lses = torch.stack([dw.lse] * cp[0])
        merged = torch.empty_like(dw.out)
        mlse = torch.empty_like(dw.lse)

        def mstep():
            bkv.bkv_merge_attn_states(outs, lses, merged, mlse, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(3):
                mstep()
        torch.cuda.synchronize()
        mg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(mg, stream=stream):
            mstep()
        mms = statistics.median(_time_steps(torch, mg.replay, max(args.steps, 20), flush, stream))
        mbytes = (outs.numel() * outs.element_size() + lses.numel() * 4 + merged.numel() * merged.element_size()
                  + mlse.numel() * 4)
        cp_merge = {"parts": cp[0], "rows": int(dw.lse.numel()), "ms": mms, "bytes": mbytes,
                    "GB_per_s": mbytes / (mms / 1e3) / 1e9, "kernel": "bkv_merge_attn_states (CUDA graph)"}

    # secondary half of the metric: slot mapping + cache write on the ragged mixed step
    secondary = None
    if rank == 0 and not args.no_secondary and headline:
        rw = wl.make("ragged_step")
        rdw = DeviceWorkload(rw, device=f"cuda:{local}", fill_prior=False)

        def wstep():
            rdw.write_step(stream=stream, fused=True)

        def wpair():
            rdw.write_step(stream=stream, fused=False)

        with torch.cuda.stream(stream):
            for _ in range(3):
                wstep()
                wpair()
        torch.cuda.synchronize()
        wbody, pbody = wstep, wpair
        if not args.eager:
            wg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(wg, stream=stream):
                wstep()
            pg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(pg, stream=stream):
                wpair()
            wbody, pbody = wg.replay, pg.replay
        reps = max(args.steps, 20)
        wm = statistics.median(_time_steps(torch, wbody, reps, flush, stream))
        pm = statistics.median(_time_steps(torch, pbody, reps, flush, stream))
        wme = statistics.median(_time_steps(torch, wstep, reps, flush, stream))
        secondary = {"workload": f"ragged_step: {rw.num_tokens} tokens of 64 requests, bs 16, H_kv 8, D 128, bf16",
                     "tokens_per_s": rw.num_tokens / (wm / 1e3), "GB_per_s": rdw.write_bytes() / (wm / 1e3) / 1e9,
                     "ms_per_step": wm, "eager_ms_per_step": wme, "kernels_per_step": 1,
                     "call": "bkv_slot_mapping_cache_write",
                     "two_calls_ms_per_step": pm, "two_calls_tokens_per_s": rw.num_tokens / (pm / 1e3),
                     "cuda_graph": not args.eager}
        del rdw

    # the other workloads, read variants and the mixed-step attention, each timed on its own
    extra, ragged = None, None
    if rank == 0 and headline and not args.no_extra:
        extra = []
        for name, window, use_fp8, cpx in EXTRA_DECODE_LEGS:
            leg = decode_leg(torch, f"cuda:{local}", flush, stream, args.steps, name, window,
                             FP8_SCALES if use_fp8 else None, cpx, args.eager)
            leg.update({"sliding_window": window, "kv_cache": "e4m3" if use_fp8 else "bf16", "cp_world": cpx[0]})
            extra.append(leg)
        ragged = ragged_leg(torch, f"cuda:{local}", flush, stream, args.steps, args.eager)

    if rank != 0:
        return
    peak, peak_kind = _peaks()
    # library kernels per timed body: block expansion; the write (one fused kernel, or slot mapping + write
    # under context parallelism); the decode (partition + merge, after the query split with FP8 caches)
    kwrite = 1 if cp[0] == 1 else 2
    kdec = 3 if fp8 is not None else 2
    kpart = kdec if cp[0] > 1 else kdec - 1
    kstep = 1 + kwrite + kdec
    achieved = kv_bytes / (pms / 1e3) / 1e9
    value = world * kv_bytes / (ms / 1e3) / 1e9
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if fp8 is None else "e4m3 cache, bf16 MMA", "data": "synthetic",
        "config": {"workload": _describe(w, args.sliding_window, cp, fp8),
                   "kv_bytes_per_step": kv_bytes, "l2": "flushed before every timed step (write 2x L2, read it back)",
                   "parallelism": f"replicas x{world}",
                   "step": ("expand + fused slot map & write + decode + merge" if kwrite == 1
                            else "expand + slot map + write + decode + merge"),
                   "cuda_graph": bool(graphs)},
        # library kernels in the timed region: per step the step, the decode alone, the partition alone and
        # the end-to-end step, plus the eager pass of the step when graphs are used
        "gpu_launches": args.steps * (2 * kstep + kdec + kpart) + (args.steps * kstep if graphs else 0),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _profiled_traffic() if headline else None,
                     "kernel": ("decode partition kernel (bkv_paged_decode_partition, CUDA events around it)"
                                if cp[0] == 1 else "context-parallel rank's decode call (partition + merge)")
                               + (": the CUDA-core kernel, forced" if args.decode_kernel == "generic" else ""),
                     "decode_call_GBps": kv_bytes / (dms / 1e3) / 1e9,
                     "peak_kind": f"{peak_kind} copy bandwidth"},
        "decode_ms": dms,
        "partition_ms": pms,
        "eager_ms_per_step": eager_ms,
        "e2e": {"value": world * kv_bytes / (ems / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes, "ms_per_step": ems},
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if secondary:
        line["secondary"] = secondary
    if headline:
        line["config4_bytes"] = bucket_report(wl.make("long_context"))
    if extra:
        line["other_workloads"] = extra
    if ragged:
        line["ragged_attention"] = ragged
    if cp_merge:
        line["cp_merge_states"] = cp_merge
    if not args.no_cpu_baseline and fp8 is None:
        line["cpu_baseline"] = _cpu_baseline(args.cpu_budget, args.workload, args.sliding_window)
    print(json.dumps(line), flush=True)


def ragged_leg(torch, dev, flush, stream, steps, eager=False, loud=False):
    """Paged attention over the mixed ragged_step batch (48 decode tokens and 16 prefill chunks of 64..1024
    tokens over prior contexts of 0..2048, H_q 32, H_kv 8, D 128, kernel bs 16, bf16), one
    bkv_paged_attention_ragged call per step, CUDA graph, L2 flushed before each step.  Prefill dominates,
    so the roofline is the tensor one: algorithmic FLOPs = 4 * D per visible (query head, key) pair."""
    from paged_kv_cache_slot_gb300 import bkv
    from paged_kv_cache_slot_gb300 import workloads as wl
    from paged_kv_cache_slot_gb300.staging import DeviceWorkload

    w = wl.make("ragged_step", loud=loud)
    dw = DeviceWorkload(w, device=dev)
    dw.write_step()
    q = torch.from_numpy(w.q_tokens()).view(torch.bfloat16).to(dev)
    out = torch.empty_like(q)
    qsl = torch.from_numpy(w.query_start_loc()).to(dev)
    mq = int(w.new_tokens.max())
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        bkv.bkv_paged_attention_ragged(q, qsl, dw.k_cache, dw.v_cache, dw.kernel_table, dw.context_lens,
                                       dw.max_context_len, mq, out, err_count=err, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    body = step
    if not eager:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        body = g.replay
    times = _time_steps(torch, body, steps, flush, stream)
    ms = sum(times) / len(times)
    assert int(err.item()) == 0
    L = w.context_lens.astype(np.int64)
    n = w.new_tokens.astype(np.int64)
    # token i of request r sees L - n + i + 1 keys: sum over i = n (L - n) + n (n + 1) / 2
    pairs = int((n * (L - n) + n * (n + 1) // 2).sum()) * w.num_q_heads
    flops = 4 * w.head_dim * pairs
    kv_bytes = int(L[n > 0].sum()) * 2 * w.num_kv_heads * w.head_dim * 2
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        peak = float(json.load(f)["bf16_tflops"])
    achieved = flops / (ms / 1e3) / 1e12
    return {"workload": f"ragged_step: {w.num_tokens} query tokens of 64 requests (48 x 1, 16 x 64..1024), prior "
                        "0..2048, H_q 32, H_kv 8, D 128, bs 16, bf16, causal",
            "ms_per_step": ms, "attended_pairs": pairs, "flops_per_step": flops, "kv_bytes_once": kv_bytes,
            "TFLOPs": achieved, "peak_TFLOPs": peak, "frac": achieved / peak,
            "peak_kind": "measured bf16 dense (burst)", "kv_GBps_once": kv_bytes / (ms / 1e3) / 1e9,
            "kernel": "bkv_paged_attention_ragged (tcgen05 prefill kernel)", "cuda_graph": not eager}


def run_ragged(args):
    """--attention ragged: the ragged leg alone, as its own JSON line (tensor roofline)."""
    import torch

    from paged_kv_cache_slot_gb300 import bkv
    from paged_kv_cache_slot_gb300.build import build

    dist = _dist()
    rank = dist.get_rank() if dist else 0
    world = dist.get_world_size() if dist else 1
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if rank == 0:
        build()
    if dist:
        dist.barrier()
    bkv.load()
    dev = f"cuda:{local}"
    stream = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = torch.empty(2 * max(l2, 64 << 20), dtype=torch.uint8, device=dev)
    if dist:
        dist.barrier()
    with ClockSampler(local) as clk:
        leg = ragged_leg(torch, dev, flush, stream, args.steps, args.eager)
    ms, = max_over_ranks([leg["ms_per_step"]], dist, dev)
    if rank != 0:
        return
    achieved = leg["flops_per_step"] / (ms / 1e3) / 1e12
    line = {
        "metric": "mixed-step paged attention TFLOP/s (ragged_step)", "value": world * achieved, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": 3, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": leg["workload"], "attended_pairs": leg["attended_pairs"],
                   "flops_per_step": leg["flops_per_step"], "kv_bytes_once": leg["kv_bytes_once"],
                   "l2": "flushed before every timed step (write 2x L2, read it back)",
                   "cuda_graph": leg["cuda_graph"]},
        "gpu_launches": args.steps,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": leg["peak_TFLOPs"], "unit": "TFLOP/s",
                     "frac": achieved / leg["peak_TFLOPs"], "traffic": None, "kernel": leg["kernel"],
                     "peak_kind": leg["peak_kind"], "kv_GBps_once": leg["kv_GBps_once"]},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def decode_leg(torch, dev, flush, stream, steps, name, window=0, fp8=None, cp=(1, 0, 1), eager=False):
    """Device times of one workload's decode, outside the headline's timed region: the partition kernel
    alone and the whole decode call (partition + merge), each a CUDA graph replayed after an L2 flush;
    the caches hold device-drawn values (timing does not depend on them)."""
    from paged_kv_cache_slot_gb300 import workloads as wl
    from paged_kv_cache_slot_gb300.staging import DeviceWorkload

    w = wl.make(name)
    dw = DeviceWorkload(w, device=dev, sliding_window=window, kv_fp8=fp8, cp_world=cp[0], cp_rank=cp[1],
                        cp_interleave=cp[2], prior_values="device")
    dw.write_step()
    kv = dw.decode_kv_bytes()

    def dec():
        dw.decode(stream=stream)

    def part():
        dw.decode_partition(stream=stream) if cp[0] == 1 else dw.decode(stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            dec()
            part()
    torch.cuda.synchronize()
    bodies = {"decode": dec, "partition": part}
    if not eager:
        for k, fn in list(bodies.items()):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            bodies[k] = g.replay
    dms = statistics.mean(_time_steps(torch, bodies["decode"], steps, flush, stream))
    pms = statistics.mean(_time_steps(torch, bodies["partition"], steps, flush, stream))
    assert int(dw.err_count.item()) == 0
    peak, _ = _peaks()
    out = {"workload": _describe(w, window, cp, fp8), "kv_bytes": kv, "partition_us": 1e3 * pms,
           "decode_call_us": 1e3 * dms, "partition_GBps": kv / (pms / 1e3) / 1e9,
           "decode_call_GBps": kv / (dms / 1e3) / 1e9}
    out["partition_frac"] = out["partition_GBps"] / peak
    out["decode_call_frac"] = out["decode_call_GBps"] / peak
    del dw
    torch.cuda.empty_cache()
    return out


# the other workloads and read variants timed beside the headline: (name, sliding window, FP8 cache,
# context-parallel (world, rank, interleave))
EXTRA_DECODE_LEGS = [
    ("long_context", 0, False, (1, 0, 1)),
    ("hybrid_spec", 0, False, (1, 0, 1)),
    ("llama3_decode", 1024, False, (1, 0, 1)),
    ("long_context", 4096, False, (1, 0, 1)),
    ("hybrid_spec", 512, False, (1, 0, 1)),
    ("llama3_decode", 0, True, (1, 0, 1)),
    ("long_context", 0, True, (1, 0, 1)),
    ("hybrid_spec", 0, True, (1, 0, 1)),
    ("llama3_decode", 0, False, (2, 0, 1)),
    ("llama3_decode", 0, False, (4, 0, 1)),
]


def run_write(args):
    """--part write: the other half of the metric alone, slot mapping + K/V cache write of the ragged
    mixed step (ragged_step: 9691 tokens of 64 requests, 48 x 1 + 16 x 64..1024, kernel bs 16, H_kv 8,
    D 128, bf16) as one bkv_slot_mapping_cache_write call per step, CUDA graph, L2 flushed before each
    step.  HBM-bound: algorithmic bytes = per token the K and V rows read and written plus its request
    index, position and slot (DeviceWorkload.write_bytes)."""
    import torch

    from paged_kv_cache_slot_gb300 import bkv
    from paged_kv_cache_slot_gb300 import workloads as wl
    from paged_kv_cache_slot_gb300.build import build
    from paged_kv_cache_slot_gb300.staging import DeviceWorkload

    dist = _dist()
    rank = dist.get_rank() if dist else 0
    world = dist.get_world_size() if dist else 1
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if rank == 0:
        build()
    if dist:
        dist.barrier()
    bkv.load()
    dev = f"cuda:{local}"
    w = wl.make("ragged_step")
    dw = DeviceWorkload(w, device=dev, fill_prior=False)
    stream = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = torch.empty(2 * max(l2, 64 << 20), dtype=torch.uint8, device=dev)

    def step():
        dw.write_step(stream=stream, fused=True)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    torch.cuda.synchronize()
    body = step
    if not args.eager:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        body = g.replay
    if dist:
        dist.barrier()
    with ClockSampler(local) as clk:
        times = _time_steps(torch, body, args.steps, flush, stream)
    ms, = max_over_ranks([sum(times) / len(times)], dist, dev)
    assert int(dw.err_count.item()) == 0
    if rank != 0:
        return
    peak, peak_kind = _peaks()
    nbytes = dw.write_bytes() + w.num_tokens * 12      # + request index and position read per token
    achieved = nbytes / (ms / 1e3) / 1e9
    line = {
        "metric": "slot-map+cache-write tokens/s (ragged_step)", "value": world * w.num_tokens / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"ragged_step: {w.num_tokens} tokens of 64 requests (48 x 1, 16 x 64..1024), prior "
                               "0..2048, kernel bs 16, H_kv 8, D 128, bf16",
                   "bytes_per_step": nbytes, "l2": "flushed before every timed step (write 2x L2, read it back)",
                   "cuda_graph": not args.eager},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "kernel": "bkv_slot_mapping_cache_write (slot_write_vec16_kernel)",
                     "peak_kind": f"{peak_kind} copy bandwidth"},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="bkv", choices=["bkv", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads, read variants and mixed-step attention timed beside the headline")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of CUDA graphs")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="seeded workload to time (default: the Llama-3-8B-shaped decode batch)")
    ap.add_argument("--sliding-window", type=int, default=0, help="decode with this sliding window (0: none)")
    ap.add_argument("--attention", default="decode", choices=["decode", "ragged"],
                    help="decode: the headline decode step; ragged: attention over the mixed ragged_step batch")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="cache element type: bf16, or E4M3 codes with per-tensor scales (bkv_*_fp8 calls)")
    ap.add_argument("--cp-world", type=int, default=1,
                    help="time rank 0 of a decode-context-parallel split over this many ranks (1: none)")
    ap.add_argument("--cp-interleave", type=int, default=1, help="context-parallel interleave size")
    ap.add_argument("--decode-kernel", default="auto", choices=["auto", "generic"],
                    help="auto: the library's choice; generic: force the CUDA-core partition kernel (comparison)")
    ap.add_argument("--part", default="step", choices=["step", "write"],
                    help="step: the whole path (default); write: slot mapping + cache write of the ragged step alone")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        if args.part == "write":
            run_write(args)
        else:
            run_ragged(args) if args.attention == "ragged" else run_bkv(args)
    d = _dist()
    if d:
        d.destroy_process_group()


if __name__ == "__main__":
    main()
