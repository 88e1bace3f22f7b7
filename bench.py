"""Benchmark: sparse MLA attention over a paged KV cache on GB300.

Default workload: MTP decode, B=64 S1=2 N_Q=128 topk=2048, act_seq 8192 for
every batch entry, 4096 shuffled 128-row blocks, bf16 cache (seeded synthetic
N(0,1) data).  One step = one call of the fused kernel over the whole batch.

  python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]
                  [--workload NAME]

``--workload indexer_decode`` (or another indexer workload) times the
Lightning Indexer + top-k instead: B=64 S1=2, 64 heads x 128 dims, 8192 keys
per sequence, top-2048; one step = one mla_indexer_topk call (the score kernel, then the
selection kernel as a programmatic dependent launch).
``--workload cache_write_decode`` / ``cache_write_prefill`` time the paged
cache writer (128 / 4096 new rows quantised into an INT8 cache of 4096 blocks).
``--workload prolog_decode`` / ``prolog_prefill`` time the MLA Prolog (128 /
1000 tokens, hidden 7168, q_lora 1536, 128 heads, random-init weights): one
step = one mla_prolog call (five launches of the library's kernels: three of
its tcgen05 product kernel and two row kernels).

Prints one JSON line (rank 0).  ``value`` is microseconds per call (the
median over the timed calls, the mean beside it; the device-timed kernel, CUDA events on the launching stream, L2 flushed by a
256 MiB write between timed calls); ``e2e`` is the same call made through the
C ABI with the step's inputs copied from pinned host memory and the outputs
copied back inside the timed region.  For the attention workloads it is
measured two ways, in order on one stream per step and as a pipelined serving
loop (copies on their own streams, double-buffered, overlapping the
neighbouring steps' calls, the L2 flush inside every step); ``e2e.value`` is
the lower, ``e2e.mode`` names it and both figures are printed.  Under torchrun every rank runs its own
batch (weak scaling, no collective on the data path); the reported time is
the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "sparse MLA attn µs/call, gathered-KV TB/s & % roofline (B64 S1=2 topk2048)"
UNIT = "us/call"
KERNEL_NAME = "mla_sparse_fwd_kernel"
KERNEL_SOURCE = os.path.join(ROOT, "mla_sparse_top_gb300", "csrc", "mla_sparse_fwd.cu")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mtp_decode",
                    choices=sorted(workloads.NAMED) + sorted(workloads.COMPRESSED_NAMED)
                    + sorted(workloads.INDEXER_NAMED)
                    + sorted(workloads.CACHE_WRITE_NAMED) + sorted(workloads.PROLOG_NAMED))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle sample")
    return ap.parse_args()


# ------------------------------------------------------------------ accounting
def row_bytes(inp):
    return (512 + 4 * 4 + 128) if inp["dims"]["kv_int8"] else (1024 + 128)


def window_positions(inp):
    """For the sliding-window workload: each token's window positions (the
    same rule as the window entry point), used only to count bytes and flops."""
    d = inp["dims"]
    W = inp["window"]
    act = np.repeat(inp["act_seqs"].astype(np.int64), d["S1"])
    p = act - d["S1"] + np.tile(np.arange(d["S1"]), d["B"])
    lists = p[:, None] - W + 1 + np.arange(W)[None, :]
    return np.where(lists >= 0, lists, -1)


def valid_mask(inp):
    d = inp["dims"]
    act = np.repeat(inp["act_seqs"], d["S1"])[:, None]
    tk = inp["topk_idx"]
    return (tk >= 0) & (tk < act)


def compressed_counts(inp):
    """CFA / SCFA accounting: per sequence the unique rows of both caches its
    tokens attend to (the window and visibility rules of the compressed entry
    point), times the row bytes, plus the per-call I/O; flops per attended
    entry as for the sparse attention."""
    d = inp["dims"]
    S1, H, W, r = d["S1"], d["n_q"], d["window"], d["cmp_ratio"]
    rb = row_bytes(inp)
    uniq, n_entries = 0, 0
    for b in range(d["B"]):
        act = int(inp["act_seqs"][b])
        ori, cmpset = set(), set()
        for s in range(S1):
            p = act - S1 + s
            win = range(max(0, p - W + 1), p + 1)
            ori.update(win)
            if "cmp_idx" in inp:
                vis = [int(i) for i in inp["cmp_idx"][b * S1 + s] if i >= 0 and (int(i) + 1) * r - 1 <= p]
            else:
                vis = list(range(0, max(0, (p + 1) // r)))
            cmpset.update(vis)
            n_entries += len(win) + len(vis)
        uniq += len(ori) + len(cmpset)
    T = d["B"] * S1
    io = T * H * (512 + 64) * 2 + T * H * 512 * 2 + T * H * 4 + inp["block_table"].nbytes + inp["act_seqs"].nbytes \
        + inp["cmp_block_table"].nbytes + (inp["cmp_idx"].nbytes if "cmp_idx" in inp else 0)
    return dict(n_valid=n_entries, gathered_bytes=n_entries * rb, roofline_bytes=uniq * rb + io,
                flops=2.0 * H * n_entries * (576 + 512))


def algorithmic_counts(inp):
    """Method's own work: counts from the actual inputs."""
    if "cmp_ratio" in inp["dims"]:
        return compressed_counts(inp)
    if "window" in inp:
        inp = dict(inp, topk_idx=window_positions(inp).astype(np.int32),
                   dims=dict(inp["dims"], topk=int(inp["window"])))
    d = inp["dims"]
    T, H = d["B"] * d["S1"], d["n_q"]
    vm = valid_mask(inp)
    n_valid = int(vm.sum())
    rb = row_bytes(inp)
    # unique physical rows touched, per batch entry (tokens of one batch entry share rows)
    uniq = 0
    for b in range(d["B"]):
        sel = inp["topk_idx"][b * d["S1"]:(b + 1) * d["S1"]][vm[b * d["S1"]:(b + 1) * d["S1"]]]
        uniq += int(np.unique(sel).size)
    io = T * H * (512 + 64) * 2 + T * H * 512 * 2 + T * H * 4 + T * d["topk"] * 4 + inp["block_table"].nbytes \
        + inp["act_seqs"].nbytes
    return dict(n_valid=n_valid, gathered_bytes=n_valid * rb, roofline_bytes=uniq * rb + io,
                flops=2.0 * H * n_valid * (576 + 512))


def roofline_of(counts, us, hbm_gbs, bf16_tf, peak_src, traffic):
    """The attention kernel's roofline object: whichever of the algorithmic bytes at the measured HBM
    bandwidth and the algorithmic FLOPs at the measured bf16 tensor peak takes longer is the bound."""
    t_bytes = counts["roofline_bytes"] / (hbm_gbs * 1e9)
    t_flops = counts["flops"] / (bf16_tf * 1e12)
    measured = peak_src == "measured"
    if t_flops > t_bytes:
        achieved = counts["flops"] / (us * 1e-6) / 1e12
        return {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16_tf, "unit": "TFLOP/s",
                "frac": round(achieved / bf16_tf, 4), "traffic": traffic,
                "peak_source": ("measured (MEASURED_PEAKS.json bf16_tflops, burst: the kernel is timed alone; "
                                "bf16 MMAs)") if measured else "fallback",
                "algorithmic_flops_per_launch": counts["flops"],
                "algorithmic_bytes_per_launch": counts["roofline_bytes"], "kernel": KERNEL_NAME}
    achieved = counts["roofline_bytes"] / (us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_gbs, "unit": "GB/s",
            "frac": round(achieved / hbm_gbs, 4), "traffic": traffic,
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if measured else "fallback",
            "algorithmic_bytes_per_launch": counts["roofline_bytes"], "kernel": KERNEL_NAME}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


INDEXER_SOURCE = os.path.join(ROOT, "mla_sparse_top_gb300", "csrc", "lightning_indexer.cu")


def kernel_source_hash(source=KERNEL_SOURCE):
    h = hashlib.sha256()
    for fn in (source, os.path.join(ROOT, "mla_sparse_top_gb300", "csrc", "ptx.cuh")):
        with open(fn, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel=KERNEL_NAME, source=KERNEL_SOURCE):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (otherwise None)."""
    fn = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(fn):
        return None
    text = open(fn).read()
    mh = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    mt = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not mh or not mt or mh.group(1) != kernel_source_hash(source):
        return None
    return float(mt.group(1))


SEEDS = {"tiny_decode": 0, "mtp_decode": 1, "int8_decode": 2, "varlen_decode": 3, "prefill": 4, "swa_decode": 10,
         "indexer_decode": 5, "indexer_tiny": 6, "indexer_varlen": 7, "cache_write_decode": 8,
         "cache_write_prefill": 9, "cfa_decode": 11, "scfa_decode": 12, "prolog_decode": 14, "prolog_prefill": 15,
         "mtp_decode_b2": 16}


def rank_seed(workload: str, rank: int) -> int:
    """Every rank draws its own batch (weak scaling): the workload's seed plus 1000 per rank."""
    return SEEDS[workload] + 1000 * rank


def pipelined_e2e(stream, flush, launch, dev, host_in, steps):
    """Microseconds per step of a serving loop through the public API: step i's
    inputs are copied from pinned host memory on an H2D stream, its call runs
    on `stream` (after the 256 MiB L2 flush, which stays inside the step), and
    its out/lse are read back to pinned host memory on a D2H stream.  Inputs
    and outputs are double-buffered, so step i's copies overlap the calls of
    steps i - 1 and i + 1; every step still copies its own inputs in and its
    own result out.  Total time from the first H2D to the last read-back,
    divided by the steps."""
    import torch
    names = list(host_in) + ["out", "lse"]
    bufs = [dict(dev), dict(dev)]
    for k in names:
        bufs[1][k] = torch.empty_like(dev[k])
    host_out = [(dev["out"].cpu().pin_memory(), dev["lse"].cpu().pin_memory()) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_call = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        j = i % 2
        b = bufs[j]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_call[j])  # the call of step i - 2 has read this input buffer
            for name, t in host_in.items():
                b[name].copy_(t, non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])  # step i - 2's result has left this output buffer
        flush.fill_(float(i))
        launch(b)
        ev_call[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_call[j])
            host_out[j][0].copy_(b["out"], non_blocking=True)
            host_out[j][1].copy_(b["lse"], non_blocking=True)
            ev_out[j].record(s_out)

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    s_in.wait_event(t0)
    for i in range(steps):
        step(i)
    stream.wait_stream(s_out)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) * 1000.0 / steps


def reduce_max_over_ranks(values, device):
    """Element-wise maximum of a list of floats over all ranks (identity when
    no process group is initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


SWA_METRIC = "sliding-window MLA attn µs/call, % HBM roofline (B64 S1=2, window 128)"


CFA_METRIC = "compressed MLA attn (CFA: window 128 + ratio-128 entries) µs/call, % HBM roofline (B64 S1=2)"
SCFA_METRIC = "sparse compressed MLA attn (SCFA: window 128 + 512 of the ratio-4 entries) µs/call, % HBM roofline (B64 S1=2)"


def metric_of(inp):
    if "cmp_ratio" in inp["dims"]:
        return SCFA_METRIC if "cmp_idx" in inp else CFA_METRIC
    return SWA_METRIC if "window" in inp else METRIC


def run_config(workload, d, world, window=None):
    """The ``config`` object of the JSON line (the same for both arms)."""
    if "cmp_ratio" in d:
        window = d["window"]
        sel = (f"window={window} + compressed ratio {d['cmp_ratio']}"
               + (f" top-{d['cmp_topk']}" if d.get("cmp_topk") else " (all visible)"))
    else:
        sel = f"window={window} (sliding)" if window else f"topk={d['topk']}"
    cfg = {
        "workload": f"{workload}: B={d['B']} S1={d['S1']} N_Q={d['n_q']} {sel} "
                    f"{'int8' if d['kv_int8'] else 'bf16'} paged cache ({d['num_blocks']} blocks of 128)",
        "B": d["B"], "S1": d["S1"], "n_q": d["n_q"], "topk": d["topk"],
        "kv_dtype": "int8" if d["kv_int8"] else "bf16",
        "l2": L2_NOTE,
        "launch": "a bounded GPU spin precedes each timed call, so its events time the device, not the host launch",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }
    if window:
        cfg["window"] = window
        del cfg["topk"]
    if "cmp_ratio" in d:
        cfg.update(cmp_ratio=d["cmp_ratio"], cmp_topk=d.get("cmp_topk") or None)
    return cfg


# ------------------------------------------------------------------ timing helpers
SPIN_CYCLES = 400_000  # about 0.2 ms of GPU time


def spin_gpu():
    """A bounded GPU spin (torch's sleep kernel) enqueued after the L2 flush, so
    that the host has enqueued the timed launch before its start event fires:
    the per-call events then measure device time, not the host's launch cost
    (which ``e2e`` includes)."""
    import torch
    torch.cuda._sleep(SPIN_CYCLES)


class L2Flush:
    """The flush between timed calls (outside their events): a 256 MiB write,
    twice L2, which evicts every line the previous call left.  ``w`` is the
    same write, used inside the pipelined serving loop's steps."""

    def __init__(self):
        import torch
        self.w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    def __call__(self, i):
        self.w.fill_(float(i))


L2_NOTE = "flushed between timed calls by a 256 MiB write (outside the per-call events)"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return self.summary()

    def summary(self):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if self.t_on is not None and self.t_on - 0.05 <= r[0] <= (self.t_off or 1e30) + 0.05]
        use = inside if inside else rows[-3:]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        mhz = [float(p[1]) for _, p in use if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for _, p in use if p[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in use:
            for k, name in enumerate(names):
                if p[5 + k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(mhz)) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(use), "in_timed_region": bool(inside)}


# ------------------------------------------------------------------ CPU oracle sample
def oracle_call(inp, tokens=None):
    """The oracle for this workload: the sliding-window oracle when it has a
    window, the sparse-attention oracle otherwise."""
    import oracle
    if "cmp_ratio" in inp["dims"]:
        import oracle.compressed as comp
        d = inp["dims"]
        return comp.forward(inp, d["window"], d["cmp_ratio"], cmp_idx=inp.get("cmp_idx"), tokens=tokens)
    if "window" in inp:
        return oracle.swa_forward(inp, inp["window"], tokens=tokens)
    return oracle.forward(inp, tokens=tokens)


def time_oracle(inp, target_s: float):
    """Time the oracle, as it stands, on a bounded token sample; returns
    (us per full call, cores, sample description)."""
    import oracle
    oracle.build()
    T = inp["dims"]["B"] * inp["dims"]["S1"]
    cores = oracle.max_threads()
    # one token per thread: the time of one parallel wave
    wave = min(T, cores)
    t0 = time.perf_counter()
    oracle_call(inp, tokens=list(range(wave)))
    t_wave = max(time.perf_counter() - t0, 1e-6)
    full_est = t_wave * math.ceil(T / wave)
    if full_est <= target_s:
        reps = max(1, int(round(target_s / full_est)))
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle_call(inp)
        dt = time.perf_counter() - t0
        return dt / reps * 1e6, cores, f"all {T} tokens, {reps} oracle calls ({dt:.2f} s)"
    n = int(min(T, max(wave, round(target_s / t_wave) * wave)))
    t0 = time.perf_counter()
    oracle_call(inp, tokens=list(range(n)))
    dt = time.perf_counter() - t0
    return dt / n * T * 1e6, cores, f"first {n} of {T} tokens in one oracle call ({dt:.2f} s), scaled to all {T} tokens"


# ------------------------------------------------------------------ main
def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if args.workload in workloads.INDEXER_NAMED:
            return run_reference_indexer(args, world, rank)
        if args.workload in workloads.CACHE_WRITE_NAMED:
            return run_reference_cache_write(args, world, rank)
        if args.workload in workloads.PROLOG_NAMED:
            return run_reference_prolog(args, world, rank)
        return run_reference(args, world, rank)
    if args.workload in workloads.INDEXER_NAMED:
        return main_indexer(args, world, rank, local_rank)
    if args.workload in workloads.CACHE_WRITE_NAMED:
        return main_cache_write(args, world, rank, local_rank)
    if args.workload in workloads.PROLOG_NAMED:
        return main_prolog(args, world, rank, local_rank)

    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    import mla_sparse_top_gb300 as mla
    from mla_sparse_top_gb300 import build
    build.build()
    mla.load_library()

    # every rank draws its own batch (weak scaling)
    gen = workloads.NAMED.get(args.workload) or workloads.COMPRESSED_NAMED[args.workload]
    inp = gen(seed=rank_seed(args.workload, rank))
    counts = algorithmic_counts(inp)
    dev = workloads.to_device(inp)
    dims = mla.dims_from_workload(inp["dims"])
    stream = torch.cuda.current_stream()
    mode = inp.get("mode", "decode")

    window = inp.get("window")
    cd = inp["dims"] if "cmp_ratio" in inp["dims"] else None
    if cd is not None:
        def _bf(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

        def _raw(a):
            return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()

        dev.update(cmp_nope=_raw(inp["cmp_nope"]) if cd["kv_int8"] else _bf(inp["cmp_nope"]),
                   cmp_rope=_bf(inp["cmp_rope"]), cmp_scales=_raw(inp.get("cmp_scales")),
                   cmp_block_table=_raw(inp["cmp_block_table"]), cmp_idx=_raw(inp.get("cmp_idx")))

    def launch(b=None):
        b = dev if b is None else b
        if cd is not None:
            mla.mla_compressed_attn_fwd(b["q_nope"], b["q_rope"], b["kv_nope"], b["kv_rope"],
                                        b["kv_scales"], b["block_table"], b["cmp_nope"], b["cmp_rope"],
                                        b["cmp_scales"], b["cmp_block_table"], b["act_seqs"], b["out"],
                                        b["lse"], window=cd["window"], cmp_ratio=cd["cmp_ratio"],
                                        cmp_idx=b["cmp_idx"], softmax_scale=inp["softmax_scale"], mode=mode,
                                        dims=dims, stream=stream)
        elif window:
            mla.mla_swa_fwd(b["q_nope"], b["q_rope"], b["kv_nope"], b["kv_rope"], b["kv_scales"],
                            b["block_table"], b["act_seqs"], b["out"], b["lse"], window=window,
                            softmax_scale=inp["softmax_scale"], mode=mode, dims=dims, stream=stream)
        else:
            mla.mla_sparse_attn_fwd(b["q_nope"], b["q_rope"], b["kv_nope"], b["kv_rope"], b["kv_scales"],
                                    b["topk_idx"], b["block_table"], b["act_seqs"], b["out"], b["lse"],
                                    softmax_scale=inp["softmax_scale"], mode=mode, dims=dims, stream=stream)

    flush = L2Flush()
    for i in range(max(3, args.warmup)):
        flush(i)
        launch()
    torch.cuda.synchronize()
    if mla.device_status(clear=True):
        raise RuntimeError("device status reported an error during warm-up")

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.15)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark_on()
    launches0 = mla.launch_count()
    for i in range(args.steps):
        flush(i)
        spin_gpu()
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    launches = mla.launch_count() - launches0
    torch.cuda.synchronize()
    clocks.mark_off()
    if world > 1:
        dist.barrier()
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    status = mla.device_status(clear=True)
    # warm: the same call back to back with no flush in between (L2 keeps what fits)
    n_warm = 20
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launch()
    w0.record(stream)
    for _ in range(n_warm):
        launch()
    w1.record(stream)
    torch.cuda.synchronize()
    warm_us = w0.elapsed_time(w1) * 1000.0 / n_warm

    # end-to-end through the C ABI with host buffers (pinned), copies inside the timed region
    per_call = ["q_nope", "q_rope", "block_table", "act_seqs"]
    if cd is not None:
        per_call += ["cmp_block_table"] + (["cmp_idx"] if dev.get("cmp_idx") is not None else [])
    elif not window:
        per_call.append("topk_idx")
    host_in = {k: dev[k].cpu().pin_memory() for k in per_call}
    host_out = dev["out"].cpu().pin_memory()
    host_lse = dev["lse"].cpu().pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out.numel() * host_out.element_size() + host_lse.numel() * host_lse.element_size()
    e2e_steps = max(5, min(args.steps, 50))
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps + 2):
        flush(i)
        k = i - 2
        if k >= 0:
            e_s[k].record(stream)
        for name, t in host_in.items():
            dev[name].copy_(t, non_blocking=True)
        launch()
        host_out.copy_(dev["out"], non_blocking=True)
        host_lse.copy_(dev["lse"], non_blocking=True)
        if k >= 0:
            e_e[k].record(stream)
    torch.cuda.synchronize()
    e2e_ms = [s.elapsed_time(e) for s, e in zip(e_s, e_e)]
    pipe_us = pipelined_e2e(stream, flush.w, launch, dev, host_in, e2e_steps)
    clock_summary = clocks.stop()

    # median of the cold-L2 calls (the headline); mean and the warm back-to-back figure beside it
    us = float(np.median(times_ms) * 1000.0)
    mean_us = float(np.mean(times_ms) * 1000.0)
    e2e_us = float(np.median(e2e_ms) * 1000.0)
    us, e2e_us, mean_us, warm_us, pipe_us = reduce_max_over_ranks([us, e2e_us, mean_us, warm_us, pipe_us],
                                                                  device="cuda")

    if rank == 0:
        hbm_gbs, bf16_tf, peak_src = measured_peaks()
        tflops = counts["flops"] / (us * 1e-6) / 1e12
        roofline_us = max(counts["roofline_bytes"] / (hbm_gbs * 1e9), counts["flops"] / (bf16_tf * 1e12)) * 1e6
        traffic = ncu_traffic(args.workload)
        d = inp["dims"]
        line = {
            "metric": metric_of(inp),
            "value": round(us, 3),
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(us / 1000.0, 6),
            "higher_is_better": False,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": run_config(args.workload, d, world, inp.get("window")),
            "timing": {"statistic": "median of cold-L2 calls", "mean_us": round(mean_us, 3),
                       "warm_back_to_back_us": round(warm_us, 3), "l2_flush": "256 MiB write between calls"},
            "gathered_kv_tbps": round(counts["gathered_bytes"] * world / (us * 1e-6) / 1e12, 4),
            "tflops": round(tflops * world, 2),
            "roofline_us": round(roofline_us, 3),
            "roofline_frac_of_call": round(roofline_us / us, 4),
            "roofline": roofline_of(counts, us, hbm_gbs, bf16_tf, peak_src, traffic),
            "tensor": {"achieved_tflops": round(tflops, 2), "peak_tflops": bf16_tf,
                       "frac": round(tflops / bf16_tf, 4), "flops_per_launch": counts["flops"]},
            "e2e": {"value": round(min(pipe_us, e2e_us), 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h),
                    "mode": "pipelined" if pipe_us <= e2e_us else "serial",
                    "pipelined_us": round(pipe_us, 3),
                    "pipelined_mode": "serving loop: each step copies its inputs in (H2D stream) and its out/lse "
                                      "back (D2H stream), double-buffered so copies overlap the neighbouring "
                                      "steps' calls; the L2 flush stays inside each step; total time / steps",
                    "serial_us": round(e2e_us, 3),
                    "serial_mode": "copies, call and read-back in order on one stream, L2 flushed before each "
                                   "step outside its events; median per step",
                    "value_is": "the lower of the two"},
            "gpu_launches": launches,
            "clocks": clock_summary,
            "device_status": status,
        }
        if not args.no_cpu_baseline:
            cus, cores, sample = time_oracle(inp, args.cpu_seconds)
            line["cpu_baseline"] = {"value": round(cus, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "sample": sample}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------ Lightning Indexer + top-k
INDEXER_METRIC = "Lightning Indexer + top-k µs/call, % HBM roofline of the score kernel (B64 S1=2 H64 topk2048)"
INDEXER_KERNELS = ("idx_scores_kernel", "idx_topk_kernel")


def indexer_counts(inp):
    """Algorithmic bytes and flops of each of the two kernels, from the inputs:
    the score kernel reads every candidate key row once (128 bf16), q, w and
    the tables, and writes one fp32 score per (token, position); the selection
    kernel reads those scores once and writes topk indices per token."""
    d = inp["dims"]
    T, H, D = d["B"] * d["S1"], d["n_heads"], d["head_dim"]
    act = np.minimum(inp["act_seqs"].astype(np.int64), d["max_blocks_per_seq"] * d["block_size"])
    keys = int(act.sum())
    tok_keys = int(np.repeat(act, d["S1"]).sum())
    tables = inp["block_table"].nbytes + inp["act_seqs"].nbytes
    scores_bytes = keys * D * 2 + T * H * D * 2 + T * H * 4 + tables + tok_keys * 4
    select_bytes = tok_keys * 4 + T * d["topk"] * 4 + inp["act_seqs"].nbytes
    flops = 2.0 * tok_keys * H * D + 2.0 * tok_keys * H
    return {"idx_scores_kernel": dict(bytes=scores_bytes, flops=flops),
            "idx_topk_kernel": dict(bytes=select_bytes, flops=0.0)}


def indexer_config(workload, d, world):
    return {
        "workload": f"{workload}: B={d['B']} S1={d['S1']} H={d['n_heads']} D={d['head_dim']} topk={d['topk']} "
                    f"bf16 paged key cache ({d['num_blocks']} blocks of 128)",
        "B": d["B"], "S1": d["S1"], "n_heads": d["n_heads"], "head_dim": d["head_dim"], "topk": d["topk"],
        "l2": L2_NOTE,
        "launch": "a bounded GPU spin precedes each timed call, so its events time the device, not the host launch",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


def indexer_subset(inp, nb):
    """The first nb sequences of an indexer workload (same cache)."""
    d = dict(inp["dims"])
    S1 = d["S1"]
    d["B"] = nb
    return dict(inp, dims=d, q=inp["q"][:nb * S1], w=inp["w"][:nb * S1], block_table=inp["block_table"][:nb],
                act_seqs=inp["act_seqs"][:nb])


def time_indexer_oracle(inp, target_s: float):
    """The oracle (scores, then selection), as it stands, on a bounded sample of
    sequences; returns (us per full call, cores, sample description)."""
    import oracle
    oracle.build()
    d = inp["dims"]
    B, S1 = d["B"], d["S1"]
    cores = oracle.max_threads()

    def run(sub):
        sc, _ = oracle.indexer_scores(sub)
        oracle.indexer_select(sc, sub["act_seqs"], S1, d["topk"])

    wave = max(1, min(B, -(-cores // S1)))          # one token per thread
    t0 = time.perf_counter()
    run(indexer_subset(inp, wave))
    t_wave = max(time.perf_counter() - t0, 1e-6)
    full_est = t_wave * math.ceil(B / wave)
    if full_est <= target_s:
        reps = max(1, int(round(target_s / full_est)))
        t0 = time.perf_counter()
        for _ in range(reps):
            run(inp)
        dt = time.perf_counter() - t0
        return dt / reps * 1e6, cores, f"all {B} sequences, {reps} oracle calls ({dt:.2f} s)"
    n = int(min(B, max(wave, round(target_s / t_wave) * wave)))
    t0 = time.perf_counter()
    run(indexer_subset(inp, n))
    dt = time.perf_counter() - t0
    return dt / n * B * 1e6, cores, f"first {n} of {B} sequences in one oracle call ({dt:.2f} s), scaled to all {B}"


def main_indexer(args, world, rank, local_rank):
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    import mla_sparse_top_gb300 as mla
    from mla_sparse_top_gb300 import build
    build.build()
    mla.load_library()

    inp = workloads.INDEXER_NAMED[args.workload](seed=rank_seed(args.workload, rank))
    d = inp["dims"]
    counts = indexer_counts(inp)
    dev = workloads.indexer_to_device(inp)
    dims = mla.indexer_dims_from_workload(d)
    scores = torch.empty(mla.mla_indexer_workspace_bytes(dims) // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def launch_scores():
        mla.mla_indexer_scores(dev["q"], dev["w"], dev["k_cache"], dev["block_table"], dev["act_seqs"], scores,
                               dims=dims, stream=stream)

    def launch_select():
        mla.mla_indexer_select(scores, dev["act_seqs"], dev["topk_idx"], dims=dims, stream=stream)

    flush = L2Flush()
    for i in range(max(3, args.warmup)):
        flush(i)
        launch_scores()
        launch_select()
    torch.cuda.synchronize()
    if mla.indexer_device_status(clear=True):
        raise RuntimeError("indexer device status reported an error during warm-up")

    def launch_both():
        mla.mla_indexer_topk(dev["q"], dev["w"], dev["k_cache"], dev["block_table"], dev["act_seqs"],
                             dev["topk_idx"], scores, dims=dims, stream=stream)

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.15)
    # the step: the public call (score kernel, then the selection kernel as a dependent launch)
    st_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark_on()
    for i in range(args.steps):
        flush(i)
        spin_gpu()
        st_ev[i][0].record(stream)
        launch_both()
        st_ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks.mark_off()
    if world > 1:
        dist.barrier()
    step_ms = [e[0].elapsed_time(e[1]) for e in st_ev]
    t_step = float(np.median(step_ms) * 1000.0)
    mean_step = float(np.mean(step_ms) * 1000.0)
    # each kernel on its own (an event between them), for the per-kernel roofline
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush(i)
        spin_gpu()
        ev[i][0].record(stream)
        launch_scores()
        ev[i][1].record(stream)
        launch_select()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    t_scores = float(np.median([e[0].elapsed_time(e[1]) for e in ev]) * 1000.0)
    t_select = float(np.median([e[1].elapsed_time(e[2]) for e in ev]) * 1000.0)
    status = mla.indexer_device_status(clear=True)

    # end to end through the public call with pinned host buffers (the key cache stays resident)
    host_in = {k: dev[k].cpu().pin_memory() for k in ("q", "w", "block_table", "act_seqs")}
    host_out = dev["topk_idx"].cpu().pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(5, min(args.steps, 50))
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps + 2):
        flush(i)
        k = i - 2
        if k >= 0:
            e_s[k].record(stream)
        for name, t in host_in.items():
            dev[name].copy_(t, non_blocking=True)
        mla.mla_indexer_topk(dev["q"], dev["w"], dev["k_cache"], dev["block_table"], dev["act_seqs"],
                             dev["topk_idx"], scores, dims=dims, stream=stream)
        host_out.copy_(dev["topk_idx"], non_blocking=True)
        if k >= 0:
            e_e[k].record(stream)
    torch.cuda.synchronize()
    e2e_us = float(np.median([a.elapsed_time(b) for a, b in zip(e_s, e_e)]) * 1000.0)
    clock_summary = clocks.stop()
    t_step, t_scores, t_select, e2e_us, mean_step = reduce_max_over_ranks(
        [t_step, t_scores, t_select, e2e_us, mean_step], device="cuda")

    if rank == 0:
        hbm_gbs, bf16_tf, peak_src = measured_peaks()
        per_kernel = {"idx_scores_kernel": t_scores, "idx_topk_kernel": t_select}
        dom = max(per_kernel, key=per_kernel.get)
        achieved = counts[dom]["bytes"] / (per_kernel[dom] * 1e-6) / 1e9
        line = {
            "metric": INDEXER_METRIC,
            "value": round(t_step, 3),
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(t_step / 1000.0, 6),
            "higher_is_better": False,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": indexer_config(args.workload, d, world),
            "kernels_us": {k: round(v, 3) for k, v in per_kernel.items()},
            "timing": {"statistic": "median of cold-L2 calls", "mean_us": round(mean_step, 3)},
            "roofline": {
                "bound": "hbm",
                "achieved": round(achieved, 1),
                "peak": hbm_gbs,
                "unit": "GB/s",
                "frac": round(achieved / hbm_gbs, 4),
                "traffic": ncu_traffic(args.workload, dom, INDEXER_SOURCE),
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback",
                "algorithmic_bytes_per_launch": counts[dom]["bytes"],
                "kernel": dom,
            },
            "tensor": {"kernel": "idx_scores_kernel",
                       "achieved_tflops": round(counts["idx_scores_kernel"]["flops"] / (t_scores * 1e-6) / 1e12, 2),
                       "peak_tflops": bf16_tf, "flops_per_launch": counts["idx_scores_kernel"]["flops"]},
            "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h)},
            "gpu_launches": 2 * args.steps,
            "kernels_note": "kernels_us from a second loop with an event between the two launches",
            "clocks": clock_summary,
            "device_status": status,
        }
        if not args.no_cpu_baseline:
            cus, cores, sample = time_indexer_oracle(inp, args.cpu_seconds)
            line["cpu_baseline"] = {"value": round(cus, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "sample": sample}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference_indexer(args, world, rank):
    """The reference arm for an indexer workload: the oracle's scores and
    selection, as they stand, on the host cores."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    inp = workloads.INDEXER_NAMED[args.workload]()
    d = inp["dims"]
    B, S1 = d["B"], d["S1"]
    cores = oracle.max_threads()
    per_step = max(1, min(B, -(-cores // S1)))
    if args.warmup > 0:
        sub = indexer_subset(inp, 1)
        oracle.indexer_scores(sub)
    per_call = []
    for i in range(args.steps):
        b0 = (i * per_step) % B
        nb = min(per_step, B - b0)
        sub = dict(indexer_subset(dict(inp, q=inp["q"][b0 * S1:], w=inp["w"][b0 * S1:],
                                       block_table=inp["block_table"][b0:], act_seqs=inp["act_seqs"][b0:]), nb))
        t0 = time.perf_counter()
        sc, _ = oracle.indexer_scores(sub)
        oracle.indexer_select(sc, sub["act_seqs"], S1, d["topk"])
        per_call.append((time.perf_counter() - t0) / nb * B * 1e6)
    us = float(np.mean(per_call))
    sample = f"{per_step} of {B} sequences per step, scaled to all {B} sequences"
    line = {
        "metric": INDEXER_METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(us / 1000.0, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": indexer_config(args.workload, d, world),
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ paged cache writer
CACHE_METRIC = "paged MLA cache write µs/call (INT8 quantise + rope copy), % HBM roofline"


def cache_write_counts(inp):
    """Algorithmic bytes: every new row read once (bf16 nope + rope + its index)
    and written once in the cache's format."""
    d = inp["dims"]
    n = int((inp["cache_index"] >= 0).sum())
    read = n * (1024 + 128) + inp["cache_index"].nbytes
    write = n * ((512 + 16) if d["kv_int8"] else 1024) + n * 128
    return read + write


def cache_write_config(workload, d, world):
    return {
        "workload": f"{workload}: T={d['T']} new rows into a {'INT8' if d['kv_int8'] else 'bf16'} paged cache of "
                    f"{d['num_blocks']} blocks of 128",
        "T": d["T"], "kv_dtype": "int8" if d["kv_int8"] else "bf16",
        "l2": L2_NOTE,
        "launch": "a bounded GPU spin precedes each timed call, so its events time the device, not the host launch",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


def time_cache_oracle(inp, target_s: float):
    import oracle
    oracle.build()
    reps, t_used = 0, 0.0
    while t_used < target_s and reps < 1000:
        t0 = time.perf_counter()
        oracle.cache_write(inp["k_nope"], inp["k_rope"], inp["cache_index"], inp["kv_nope"], inp["kv_rope"],
                           inp["kv_scales"], inplace=True)
        t_used += time.perf_counter() - t0
        reps += 1
    return t_used / reps * 1e6, 1, f"the whole call, {reps} oracle calls ({t_used:.2f} s), writing in place"


def main_cache_write(args, world, rank, local_rank):
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    import mla_sparse_top_gb300 as mla
    from mla_sparse_top_gb300 import build
    build.build()
    mla.load_library()
    inp = workloads.CACHE_WRITE_NAMED[args.workload](seed=rank_seed(args.workload, rank))
    d = inp["dims"]
    dev = workloads.cache_write_to_device(inp)
    stream = torch.cuda.current_stream()

    def launch():
        mla.mla_cache_write(dev["k_nope"], dev["k_rope"], dev["cache_index"], dev["kv_nope"], dev["kv_rope"],
                            dev["kv_scales"], stream=stream)

    flush = L2Flush()
    for i in range(max(3, args.warmup)):
        flush(i)
        launch()
    torch.cuda.synchronize()
    if mla.cache_device_status(clear=True):
        raise RuntimeError("cache writer device status reported an error during warm-up")
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.15)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark_on()
    for i in range(args.steps):
        flush(i)
        spin_gpu()
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    torch.cuda.synchronize()
    clocks.mark_off()
    if world > 1:
        dist.barrier()
    call_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    us = float(np.median(call_ms) * 1000.0)
    mean_us = float(np.mean(call_ms) * 1000.0)
    status = mla.cache_device_status(clear=True)
    # end to end: the new rows and their indices from pinned host memory, then the call; the
    # result is the updated device cache, so nothing is read back but the status word
    host_in = {k: dev[k].cpu().pin_memory() for k in ("k_nope", "k_rope", "cache_index")}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    e2e_steps = max(5, min(args.steps, 50))
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps + 2):
        flush(i)
        k = i - 2
        if k >= 0:
            e_s[k].record(stream)
        for name, t in host_in.items():
            dev[name].copy_(t, non_blocking=True)
        launch()
        if k >= 0:
            e_e[k].record(stream)
    torch.cuda.synchronize()
    e2e_us = float(np.median([a.elapsed_time(b) for a, b in zip(e_s, e_e)]) * 1000.0)
    clock_summary = clocks.stop()
    us, e2e_us, mean_us = reduce_max_over_ranks([us, e2e_us, mean_us], device="cuda")
    if rank == 0:
        hbm_gbs, _, peak_src = measured_peaks()
        nbytes = cache_write_counts(inp)
        achieved = nbytes / (us * 1e-6) / 1e9
        line = {
            "metric": CACHE_METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(us / 1000.0, 6), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8" if d["kv_int8"] else "bf16",
            "data": "synthetic", "config": cache_write_config(args.workload, d, world),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_gbs, "unit": "GB/s",
                         "frac": round(achieved / hbm_gbs, 4), "traffic": None,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                         else "fallback",
                         "algorithmic_bytes_per_launch": nbytes, "kernel": "cache_write_kernel"},
            "timing": {"statistic": "median of cold-L2 calls", "mean_us": round(mean_us, 3)},
            "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": 0},
            "gpu_launches": args.steps, "clocks": clock_summary, "device_status": status,
        }
        if not args.no_cpu_baseline:
            cus, cores, sample = time_cache_oracle(inp, min(args.cpu_seconds, 5.0))
            line["cpu_baseline"] = {"value": round(cus, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "sample": sample}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference_cache_write(args, world, rank):
    """The reference arm for a cache-write workload: the oracle, as it stands, on one host core."""
    if rank != 0:
        return
    inp = workloads.CACHE_WRITE_NAMED[args.workload]()
    d = inp["dims"]
    import oracle
    oracle.build()
    per_call = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.cache_write(inp["k_nope"], inp["k_rope"], inp["cache_index"], inp["kv_nope"], inp["kv_rope"],
                           inp["kv_scales"], inplace=True)
        per_call.append((time.perf_counter() - t0) * 1e6)
    us = float(np.mean(per_call))
    line = {
        "metric": CACHE_METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(us / 1000.0, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
        "config": cache_write_config(args.workload, d, world),
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "the whole call per step, writing in place"},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ MLA Prolog
PROLOG_METRIC = "MLA Prolog µs/call (x -> absorbed q_nope/q_rope + cache row), % HBM roofline on weight bytes"


def prolog_counts(inp):
    """Algorithmic bytes and flops of one call: every weight, x, cos/sin and the
    indices read once; q_nope, q_rope and the cache rows written once.  The
    fp32 projections and bf16 operands kept in the workspace between launches
    are not counted (a fused kernel would not need them)."""
    d = inp["dims"]
    T, hd, ql, H = d["T"], d["hidden"], d["q_lora"], d["n_heads"]
    weights = 2 * (hd * ql + ql + ql * H * 192 + H * 128 * 512 + hd * 576 + 576)
    n = int((inp["cache_index"] >= 0).sum())
    rows = n * (((512 + 16) if d["kv_int8"] else 1024) + 128)
    nbytes = weights + 2 * T * hd + 2 * 4 * T * 32 + 8 * T + 2 * T * H * (512 + 64) + rows
    flops = 2 * T * (hd * ql + ql * H * 192 + H * 128 * 512 + hd * 576)
    return nbytes, flops


def prolog_config(workload, d, world):
    return {
        "workload": f"{workload}: T={d['T']} tokens, hidden {d['hidden']}, q_lora {d['q_lora']}, {d['n_heads']} heads "
                    f"(DeepSeek-V3.2 sizes, random-init bf16 weights), {'INT8' if d['kv_int8'] else 'bf16'} paged "
                    f"cache of {d['num_blocks']} blocks of 128",
        "T": d["T"], "hidden": d["hidden"], "q_lora": d["q_lora"], "n_heads": d["n_heads"],
        "kv_dtype": "int8" if d["kv_int8"] else "bf16",
        "l2": L2_NOTE,
        "launch": "a bounded GPU spin precedes each timed call, so its events time the device, not the host launch",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


def main_prolog(args, world, rank, local_rank):
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    import mla_sparse_top_gb300 as mla
    from mla_sparse_top_gb300 import build
    build.build()
    mla.load_library()
    inp = workloads.PROLOG_NAMED[args.workload](seed=rank_seed(args.workload, rank))
    d = inp["dims"]
    dev = workloads.prolog_to_device(inp)
    T, H = d["T"], d["n_heads"]
    q_nope = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    q_rope = torch.empty((T, H, 64), dtype=torch.bfloat16, device="cuda")
    dims = mla.prolog_dims(dev["x"], dev["wq_a"], dev["wq_b"], dev["kv_nope"])
    ws = torch.empty(mla.mla_prolog_workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def launch():
        mla.mla_prolog(dev["x"], dev["wq_a"], dev["gamma_cq"], dev["wq_b"], dev["w_uk"], dev["wkv"],
                       dev["gamma_ckv"], dev["cos"], dev["sin"], dev["cache_index"], q_nope, q_rope, dev["kv_nope"],
                       dev["kv_rope"], dev["kv_scales"], ws, dims=dims, stream=stream)

    flush = L2Flush()
    for i in range(max(3, args.warmup)):
        flush(i)
        launch()
    torch.cuda.synchronize()
    if mla.prolog_device_status(clear=True):
        raise RuntimeError("prolog device status reported an error during warm-up")
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.15)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark_on()
    for i in range(args.steps):
        flush(i)
        spin_gpu()
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    torch.cuda.synchronize()
    clocks.mark_off()
    if world > 1:
        dist.barrier()
    call_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    us = float(np.median(call_ms) * 1000.0)
    mean_us = float(np.mean(call_ms) * 1000.0)
    status = mla.prolog_device_status(clear=True)
    # end to end: x, cos/sin and the indices from pinned host memory, the call, q_nope and q_rope back
    host_in = {k: dev[k].cpu().pin_memory() for k in ("x", "cos", "sin", "cache_index")}
    h_qn = torch.empty(q_nope.shape, dtype=q_nope.dtype, pin_memory=True)
    h_qr = torch.empty(q_rope.shape, dtype=q_rope.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = h_qn.numel() * 2 + h_qr.numel() * 2
    e2e_steps = max(5, min(args.steps, 50))
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps + 2):
        flush(i)
        k = i - 2
        if k >= 0:
            e_s[k].record(stream)
        for name, t in host_in.items():
            dev[name].copy_(t, non_blocking=True)
        launch()
        h_qn.copy_(q_nope, non_blocking=True)
        h_qr.copy_(q_rope, non_blocking=True)
        if k >= 0:
            e_e[k].record(stream)
    torch.cuda.synchronize()
    e2e_us = float(np.median([a.elapsed_time(b) for a, b in zip(e_s, e_e)]) * 1000.0)
    clock_summary = clocks.stop()
    us, e2e_us, mean_us = reduce_max_over_ranks([us, e2e_us, mean_us], device="cuda")
    if rank == 0:
        hbm_gbs, bf16_tf, peak_src = measured_peaks()
        nbytes, flops = prolog_counts(inp)
        achieved = nbytes / (us * 1e-6) / 1e9
        line = {
            "metric": PROLOG_METRIC, "value": round(us, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(us / 1000.0, 6), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init weights)",
            "config": prolog_config(args.workload, d, world),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_gbs, "unit": "GB/s",
                         "frac": round(achieved / hbm_gbs, 4), "traffic": None,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                         else "fallback",
                         "algorithmic_bytes_per_launch": nbytes,
                         "kernel": "the whole mla_prolog call (gemm_kernel x3 + x_rows_kernel, q_heads_kernel)",
                         "tensor_tflops": round(flops / (us * 1e-6) / 1e12, 1),
                         "tensor_frac_of_bf16_peak": round(flops / (us * 1e-6) / 1e12 / bf16_tf, 4)},
            "timing": {"statistic": "median of cold-L2 calls", "mean_us": round(mean_us, 3)},
            "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h)},
            "gpu_launches": 5 * args.steps, "clocks": clock_summary,
            "device_status": status,
        }
        if not args.no_cpu_baseline:
            cus, sample = time_prolog_oracle(inp, min(args.cpu_seconds, 10.0))
            line["cpu_baseline"] = {"value": round(cus, 1), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                                    "sample": sample}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def time_prolog_oracle(inp, target_s: float):
    """The oracle (numpy fp64, its matrix products on numpy's BLAS threads) on
    whole calls until ``target_s`` of CPU time is used."""
    import oracle.prolog as P
    reps, t_used = 0, 0.0
    while t_used < target_s and reps < 100:
        t0 = time.perf_counter()
        P.forward_with_cache(inp)
        t_used += time.perf_counter() - t0
        reps += 1
    return t_used / reps * 1e6, (f"the whole call, {reps} oracle calls ({t_used:.2f} s); numpy BLAS threads "
                                 f"up to the host's cores")


def run_reference_prolog(args, world, rank):
    """The reference arm for a prolog workload: the oracle, as it stands, one whole call per step."""
    if rank != 0:
        return
    inp = workloads.PROLOG_NAMED[args.workload]()
    d = inp["dims"]
    import oracle.prolog as P
    for _ in range(min(args.warmup, 1)):
        P.forward_with_cache(inp)
    per_call = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        P.forward_with_cache(inp)
        per_call.append((time.perf_counter() - t0) * 1e6)
    us = float(np.mean(per_call))
    line = {
        "metric": PROLOG_METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(us / 1000.0, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (random-init weights)", "impl": "reference",
        "config": prolog_config(args.workload, d, world),
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "the whole call per step (numpy BLAS threads up to the host's cores)"},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    gen = workloads.NAMED.get(args.workload) or workloads.COMPRESSED_NAMED[args.workload]
    inp = gen()
    d = inp["dims"]
    T = d["B"] * d["S1"]
    cores = oracle.max_threads()
    toks_per_step = max(1, cores)
    if args.warmup > 0:
        oracle_call(inp, tokens=[0])
    per_call, step_s = [], []
    for i in range(args.steps):
        toks = [(i * toks_per_step + k) % T for k in range(toks_per_step)]
        t0 = time.perf_counter()
        oracle_call(inp, tokens=toks)
        step_s.append(time.perf_counter() - t0)
        per_call.append(step_s[-1] / len(toks) * T * 1e6)
    us = float(np.mean(per_call))
    sample = f"{toks_per_step} of {T} tokens per step, scaled to all {T} tokens"
    line = {
        "metric": metric_of(inp), "value": round(us, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        # a step is the token sample; value is the whole call extrapolated from it
        "warmup": args.warmup, "ms_per_step": round(float(np.mean(step_s)) * 1000.0, 3),
        "value_kind": "per-call time extrapolated from the sampled tokens of each step",
        "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": run_config(args.workload, d, world, inp.get("window")),
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
