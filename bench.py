"""Benchmark of the paged-KV varlen attention path on GB300.

A step is one pass of the whole hot path over one batch: the KV append (slot mapping fused into
the copy kernel), paged attention and the split-KV merge, with the block table and task table
(host-built per batch) already on the device.  The default run measures the decode batch (64
sequences, q = 1, context U[128, 4096], 32/32 heads, d = 128, 16-token pages) for the headline
line, and in the same run the packed prefill, mixed continuous, long-context skew,
speculative-verify and prefix-shared batches, each under its own key with the same
measurements.  `--config` picks the headline batch, `--only` measures that one alone.

Prints one JSON line (rank 0).  Per batch: `value` is device-timed throughput of the step with
inputs resident in HBM (CUDA events around exactly `--steps` steps; L2 flushed before each step
when the batch's working set would otherwise stay in L2); `roofline` reports the attention
kernel's algorithmic bytes (or flops) over its average launch time, taken in a separate
instrumented pass, against the measured peak; `e2e` is the same metric through the public Python
API with pinned host inputs copied in and the output copied out every step; `cpu_baseline` times
the oracle on a bounded sample on the host cores; `clocks` holds the SM clock and throttle
reasons sampled during the timed steps.  `--impl reference` times the oracle alone.
Multi-GPU (torchrun): independent replicas, one per rank (weak scaling, no data-path collective).
"""

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

# the oracle baseline runs single-threaded BLAS so its core count is exact
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged-attn decode KV GB/s & prefill TFLOP/s vs roofline, tokens/s, 1×GB300"
NOMINAL = {"hbm": 8000.0, "tc": 2250.0}   # the nominal GB300 figures (GB/s, dense BF16 TFLOP/s)
DESC = {
    "tiny": "tiny mixed: 4 seqs (q 7,16,1,1; L 7,16,33,50), Hq 4 / Hkv 2, d 64, bs 16",
    "decode": "decode: 64 seqs, q=1, L~U[128,4096], Hq=Hkv=32, d=128, bs=16, + kv_append of 64 tokens",
    "prefill": "packed prefill: 16 seqs lognormal(512,1) in [32,8192], causal, Hq 32 / Hkv 8, d 128, bs 16",
    "mixed": "mixed: 8 chunks x 512 (prior U[0,16384]) + 120 decodes L~U[256,32768], Hq 32 / Hkv 8, d 128, bs 16",
    "skew": "long-context skew: 256 decodes (4 x 131072, 252 x 512), Hq 64 / Hkv 8, d 128, bs 256",
    "verify": "speculative verify: 64 seqs, q~U{2..8} over L~U[512,8192], Hq 32 / Hkv 8, d 128, bs 16",
    "prefix": "prefix-shared decode: 64 seqs x L=4096, first 3584 tokens on shared pages, Hq=Hkv=32, d 128, bs 16",
}
# measured in the default run beside the headline batch, under these keys of the JSON line
# batches measured beside the headline one: JSON key -> (batch, page format); the default (bf16)
# line also carries the decode batch over 8-bit pages
SECONDARY = {"prefill": ("prefill", "bf16"), "mixed": ("mixed", "bf16"), "skew": ("skew", "bf16"),
             "verify": ("verify", "bf16"), "prefix_shared": ("prefix", "bf16"), "decode_fp8": ("decode", "fp8")}
SECONDARY_FP8 = {"prefill": ("prefill", "fp8"), "mixed": ("mixed", "fp8"), "skew": ("skew", "fp8")}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], tc=d["bf16_tflops"], tc_sustained=d.get("bf16_tflops_sustained"),
                    source="measured")
    return dict(hbm=6800.0, tc=1900.0, tc_sustained=1700.0, source="fallback")


def measured_traffic(config):
    """DRAM bytes per attention launch from a committed ncu capture, or None when there is no
    capture for this workload or the kernel source changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get("entries", {}).get(config)
    if not e:
        return None
    h = hashlib.sha256()
    for f in d["hash_files"]:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return e["bytes_per_launch"] if h.hexdigest()[:16] == e["kernel_hash"] else None


def work(wl, kv="bf16", block_table=None):
    """Algorithmic work of one step: attention bytes (K/V read once + Q in + O out), append bytes
    (new K/V read + written), and flops (4 d per visible (row, key) pair per query head).  A stored
    K or V row is d bf16 values, or over 8-bit pages d codes and one fp32 scale.  With a block table
    whose rows share pages (prefix sharing), `unique_attn_bytes` counts each physical page once."""
    d, Hq, Hkv = wl.head_dim, wl.num_heads_q, wl.num_heads_kv
    L = wl.context_lens.astype(np.int64)
    q = wl.q_lens.astype(np.int64)
    row_bytes = d + 4 if kv == "fp8" else 2 * d
    kv_bytes = int(np.sum(L) * 2 * Hkv * row_bytes)
    qo_bytes = int(wl.num_tokens * Hq * d * 2 * 2)
    append_bytes = int(wl.num_tokens * Hkv * 2 * (2 * d + row_bytes))
    if wl.causal:
        pairs = int(np.sum(q * (L - q) + q * (q + 1) // 2))
    else:
        pairs = int(np.sum(q * L))
    flops = 4 * d * Hq * pairs
    w = dict(attn_bytes=kv_bytes + qo_bytes, append_bytes=append_bytes, flops=flops, kv_bytes=kv_bytes)
    if block_table is not None:
        # keys held by each distinct physical page (the last page of a row may be partial)
        bs = wl.block_size
        held = {}
        for i, row in enumerate(np.asarray(block_table)):
            n = -(-int(L[i]) // bs)
            for j in range(n):
                held[int(row[j])] = max(held.get(int(row[j]), 0), min(bs, int(L[i]) - j * bs))
        w["unique_attn_bytes"] = int(sum(held.values()) * 2 * Hkv * row_bytes) + qo_bytes
    return w


class NvmlClocks:
    """SM clock and clock-event (throttle) reasons read through NVML every `period_s` while
    running (reads only; nothing is set).  The GPU is found by the UUID of the CUDA device, so the
    samples belong to it whatever CUDA_VISIBLE_DEVICES maps."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, dev, period_s=0.001):
        self.period_s, self.samples, self.ok = period_s, [], False
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
            self.h = ctypes.c_void_p()
            if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
                return
            self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 \
                else None
            self.ok = True
        except (OSError, AttributeError, RuntimeError):
            self.ok = False

    def _run(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop:
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0 and \
                    self.reasons_fn(self.h, ctypes.byref(rs)) == 0:
                self.samples.append((time.perf_counter(), float(clk.value), int(rs.value)))
            time.sleep(self.period_s)

    def start(self):
        self.samples, self._stop = [], False
        if self.ok:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        return self

    def stop(self):
        self._stop = True
        if self.ok:
            self.thread.join()

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:   # a timed region shorter than one NVML read: the samples nearest to it
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
        if not inside:
            return None
        reasons = sorted({n for _, _, r in inside for b, n in self.REASONS.items() if r & b})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(inside),
                "samples_in_window": sum(1 for s in inside if t0 <= s[0] <= t1),
                "window_ms": 1e3 * (t1 - t0), "source": "NVML, every 1 ms during the timed steps"}


class SmiClocks:
    """nvidia-smi samples (every 20 ms) of SM clock and throttle reasons over the whole run (the
    query line of the profiling recipe); `summary(t0, t1)` keeps the samples inside [t0, t1]."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
        self.gpu = f"GPU-{uuid}" if uuid is not None else str(dev.index)
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ts, ln in self.lines:
            if t0 is not None and not (t0 <= ts <= t1):
                continue
            f = [x.strip() for x in ln.split(",")]
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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi every 20 ms, " +
                ("timed steps" if t0 is not None else "whole run")}


def oracle_sample(wl, vals, budget_s=12.0, max_seqs=None, kv="bf16"):
    """Time the oracle (as it stands) on a bounded sample of the workload's sequences, all their
    rows (over 8-bit pages: its 8-bit step, quantizing the sampled pages first).  Returns
    (seconds, sampled work dict, description, sampled sequences, seconds per sequence)."""
    import oracle

    def bits(t):
        return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    bt = oracle.allocate_block_table(wl.context_lens, wl.block_size, wl.free_list, wl.max_blocks)
    rng = np.random.default_rng(0)
    order = rng.permutation(wl.num_seqs)
    cu = wl.cu_seqlens_q
    spent, done, per_seq = 0.0, [], []
    q_all, kn_all, vn_all = bits(vals["q"]), bits(vals["k_new"]), bits(vals["v_new"])
    for i in order:
        if spent >= budget_s or (max_seqs and len(done) >= max_seqs):
            break
        i = int(i)
        pages = bt[i][bt[i] >= 0]
        idx = torch.from_numpy(pages).long().to(vals["k_pool"].device)
        kp, vp = bits(vals["k_pool"].index_select(0, idx)), bits(vals["v_pool"].index_select(0, idx))
        t0, t1 = int(cu[i]), int(cu[i + 1])
        sub_cu = np.array([0, t1 - t0], np.int32)
        t = time.perf_counter()
        run = oracle.step.run_step_fp8 if kv == "fp8" else oracle.step.run_step
        run(sub_cu, wl.context_lens[i:i + 1], pages, wl.block_size, wl.max_blocks, q_all[t0:t1], kn_all[t0:t1],
            vn_all[t0:t1], kp, vp, wl.scale, wl.causal, pool_pages=pages)
        per_seq.append(time.perf_counter() - t)
        spent += per_seq[-1]
        done.append(i)
    sub = workloads.custom(wl.q_lens[done], wl.context_lens[done], wl.num_heads_q, wl.num_heads_kv, wl.head_dim,
                           wl.block_size, wl.causal)
    desc = f"{len(done)} of {wl.num_seqs} sequences (seeded random order), every row, full oracle step"
    return spent, work(sub, kv), desc, done, per_seq


def oracle_sample_cores(wl, vals, seqs, seq_secs, kv="bf16"):
    """The oracle on all host cores: one single-threaded process per core (`python -m
    oracle.timing`), the sequences of the single-core sample (`seqs`, whose single-core oracle
    seconds are `seq_secs`) dealt longest-first to the least-loaded process.  Returns (the sampled
    workload, the slowest process's oracle seconds, cores, description)."""
    import tempfile
    cores = len(os.sched_getaffinity(0))

    def bits(t):
        return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    import oracle
    bt = oracle.allocate_block_table(wl.context_lens, wl.block_size, wl.free_list, wl.max_blocks)
    chosen = list(seqs)
    loads = [0.0] * cores
    parts = [[] for _ in range(cores)]
    for i, sec in sorted(zip(seqs, seq_secs), key=lambda x: -x[1]):
        c = loads.index(min(loads))
        parts[c].append(i)
        loads[c] += sec
    q_all, kn_all, vn_all = bits(vals["q"]), bits(vals["k_new"]), bits(vals["v_new"])
    cu = wl.cu_seqlens_q
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    with tempfile.TemporaryDirectory() as tmp:
        procs = []
        for c, part in enumerate(parts):
            if not part:
                continue
            arrs = {"n": len(part), "kv": kv, "bs": wl.block_size, "mb": wl.max_blocks, "scale": wl.scale,
                    "causal": int(wl.causal)}
            for k, i in enumerate(part):
                pages = bt[i][bt[i] >= 0]
                idx = torch.from_numpy(pages).long().to(vals["k_pool"].device)
                t0, t1 = int(cu[i]), int(cu[i + 1])
                arrs.update({f"cu_{k}": np.array([0, t1 - t0], np.int32), f"ctx_{k}": wl.context_lens[i:i + 1],
                             f"pages_{k}": pages, f"q_{k}": q_all[t0:t1], f"kn_{k}": kn_all[t0:t1],
                             f"vn_{k}": vn_all[t0:t1], f"kp_{k}": bits(vals["k_pool"].index_select(0, idx)),
                             f"vp_{k}": bits(vals["v_pool"].index_select(0, idx))})
            path = os.path.join(tmp, f"part{c}.npz")
            np.savez(path, **arrs)
            procs.append(subprocess.Popen([sys.executable, "-m", "oracle.timing", path], cwd=ROOT, env=env,
                                          stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
        secs = []
        for pr in procs:
            try:
                out, err = pr.communicate(timeout=300)
            except subprocess.TimeoutExpired:
                pr.kill()
                pr.communicate()
                raise RuntimeError("an oracle timing process ran past 300 s")
            if pr.returncode != 0:
                raise RuntimeError("oracle timing process failed: " + err[-500:])
            secs.append(json.loads(out.strip().splitlines()[-1])["seconds"])
    sub = workloads.custom(wl.q_lens[chosen], wl.context_lens[chosen], wl.num_heads_q, wl.num_heads_kv,
                           wl.head_dim, wl.block_size, wl.causal)
    desc = (f"the single-core sample's {len(chosen)} sequences, dealt longest-first (by their single-core "
            f"time) over {len([p for p in parts if p])} single-threaded processes; time = the slowest process's "
            f"oracle seconds")
    return sub, max(secs), cores, desc


def unit_of(config):
    return ("TFLOP/s", "tensor") if config == "prefill" else ("GB/s", "hbm")


def max_over_ranks(x, world, device="cpu"):
    """The largest of one float per rank (the slowest replica sets the job's time); `device` is
    where the reduction tensor lives ("cuda:i" under NCCL, "cpu" under gloo)."""
    if world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(config, w, seconds, world):
    """Whole-job throughput of `world` replicas that each process work `w` in `seconds` (the max
    over ranks): the units all ranks processed / that time."""
    return throughput(config, w, seconds) * world


def attention_kernel(wl, kv="bf16", schedule=3):
    """The attention kernel the library dispatches to: the tcgen05 tile kernel when head_dim is
    128, G divides 128 and the batch is not pure decode (one token per sequence, G <= 16);
    otherwise, and always over 8-bit pages, the decode-path kernel."""
    if schedule == 4:
        name = attention_kernel(wl, kv)
        G = wl.num_heads_q // wl.num_heads_kv
        if name == "paged_attention_kernel" and wl.num_tokens == wl.num_seqs and G <= (8 if kv == "fp8" else 16):
            name += ", two CTAs per SM"   # pure decode under the dynamic deal: half-size CTAs
        return name + " (dynamic deal)"
    if kv == "fp8":
        return "paged_attention_kernel"
    G = wl.num_heads_q // wl.num_heads_kv
    pure_decode = wl.num_tokens == wl.num_seqs and G <= 16
    if wl.head_dim == 128 and 128 % G == 0 and not pure_decode:
        return "meta_attention_kernel"
    return "paged_attention_kernel"


def throughput(config, w, seconds):
    if config == "prefill":
        return w["flops"] / seconds / 1e12
    return (w["attn_bytes"] + w["append_bytes"]) / seconds / 1e9


def describe(config, args):
    return (DESC[config] + (", 8-bit E4M3 KV pages + per-row fp32 scales" if args.kv == "fp8" else "") +
            (", dynamic deal (CTAs claim tasks at run time)" if args.schedule == 4 else
             f", static deal (task-table schedule {args.schedule})"))


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = workloads.make(args.config)
    vals = wl.tensors("cuda" if torch.cuda.is_available() else "cpu")
    unit, _ = unit_of(args.config)
    times = []
    for k in range(args.warmup + args.steps):
        secs, w, desc, _, _ = oracle_sample(wl, vals, budget_s=args.ref_budget, kv=args.kv)
        if k >= args.warmup:
            times.append((secs, w))
    secs = sum(t for t, _ in times)
    value = sum(throughput(args.config, w, t) * t for t, w in times) / secs if secs else 0.0
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(args.config, args)},
            "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure(config, args, dev, pk, world, rank, cpu_budget, smi):
    """Every measurement of one batch: device-timed steps, the instrumented pass (attention and
    append times), a traced launch (deal balance), the end-to-end serving loop and the oracle
    baseline.  Returns the batch's JSON object (the headline line's fields for the headline)."""
    import paged_kv_varlen_xy_gb300 as xy
    from paged_kv_varlen_xy_gb300 import step as xystep

    wl = workloads.make(config)
    vals = wl.tensors(dev)
    fp8 = args.kv == "fp8"
    # over 8-bit pages a batch with prefill / chunk sequences runs them on the tile path over bf16
    # copies of their pages and its decode sequences on the 8-bit decode path (when the two kinds
    # form contiguous sequence ranges and the tile shape allows)
    G = wl.num_heads_q // wl.num_heads_kv
    split = (fp8 and wl.num_tokens != wl.num_seqs and wl.head_dim == 128 and 128 % G == 0
             and xystep.split_ranges(wl.q_lens) is not None)
    if split:
        batch = xystep.Fp8SplitBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                                     wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, device=dev)
        parts = [x["plan"] for x in (batch.tile, batch.decode) if x is not None]
    else:
        batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                                  wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, device=dev, kv_fp8=fp8,
                                  schedule=args.schedule)
        parts = [batch.plan]
    shared_bt = None
    if wl.shared_prefix_tokens:
        # prefix sharing: every row's first pages are row 0's (the kernels read pages only through
        # the block table); the new tokens land after the prefix, in each row's own pages
        shared_bt = workloads.share_prefix(batch.block_table_host, wl.shared_prefix_tokens, wl.block_size)
        batch.block_table.copy_(torch.from_numpy(shared_bt))
        batch.block_table_host = shared_bt
    w = work(wl, args.kv, block_table=shared_bt)
    pl = parts[0]
    n_tasks = sum(int(x.tasks.shape[0]) for x in parts)
    n_merges = sum(int(x.merges.shape[0]) for x in parts)
    stream = torch.cuda.current_stream(dev)
    out = torch.empty_like(vals["q"])
    P = wl.num_pages
    if fp8:
        # the 8-bit pool: every bf16 pool row appended (quantized) once, before any timing
        Pp, Hkv, bs, d = vals["k_pool"].shape
        # K and V codes in one allocation, V after K: the attention brings a page's K and V codes
        # with one copy (separate allocations work too, with a copy per page and pool)
        codes = torch.empty(2, Pp, Hkv, bs, d, dtype=torch.uint8, device=dev)
        vals["k_codes"], vals["v_codes"] = codes[0], codes[1]
        for name in ("k", "v"):
            vals[name + "_scales"] = torch.empty(Pp, Hkv, bs, dtype=torch.float32, device=dev)
        rows = {n: vals[n + "_pool"].permute(0, 2, 1, 3).reshape(Pp * bs, Hkv, d).contiguous() for n in ("k", "v")}
        xy.xy_kv_append_fp8(rows["k"], rows["v"], torch.arange(Pp * bs, dtype=torch.int64, device=dev),
                            vals["k_codes"], vals["v_codes"], vals["k_scales"], vals["v_scales"], batch.err)
        del rows
        torch.cuda.synchronize()

    def append():
        if fp8:
            xy.xy_kv_append_paged_fp8(vals["k_new"], vals["v_new"], batch.cu, batch.ctx, batch.block_table,
                                      vals["k_codes"], vals["v_codes"], vals["k_scales"], vals["v_scales"], batch.err,
                                      slot_mapping=batch.slots)
        else:
            xy.xy_kv_append_paged(vals["k_new"], vals["v_new"], batch.cu, batch.ctx, batch.block_table,
                                  vals["k_pool"], vals["v_pool"], batch.err, slot_mapping=batch.slots)

    def attend():
        if split:
            xystep.attention_fp8_split(batch, vals["q"], vals["k_codes"], vals["v_codes"], vals["k_scales"],
                                       vals["v_scales"], wl.scale, out)
        elif fp8 and pl.dynamic:
            xy.xy_paged_attention_fp8_dynamic(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_codes"],
                                              vals["v_codes"], vals["k_scales"], vals["v_scales"], wl.scale,
                                              wl.causal, pl.tasks, pl.merges, pl.num_ctas, pl.workspace,
                                              pl.task_counter, batch.err, out)
        elif fp8:
            xy.xy_paged_attention_fp8(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_codes"],
                                      vals["v_codes"], vals["k_scales"], vals["v_scales"], wl.scale, wl.causal,
                                      pl.tasks, pl.merges, pl.num_ctas, pl.workspace, batch.err, out)
        elif pl.dynamic:
            xy.xy_paged_attention_dynamic(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"],
                                          vals["v_pool"], wl.scale, wl.causal, pl.tasks, pl.merges, pl.num_ctas,
                                          pl.workspace, pl.task_counter, batch.err, out)
        else:
            xy.xy_paged_attention(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"], vals["v_pool"],
                                  wl.scale, wl.causal, pl.tasks, pl.merges, pl.num_ctas, pl.workspace, batch.err, out)

    def step():
        append()
        attend()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    xystep.check(batch)

    # Between timed steps: a batch whose data would stay in the 129 MB L2 from one step to the next
    # gets the L2 flushed (a write of twice its size) before every step, outside the timed events;
    # larger batches run back to back.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    touched = w.get("unique_attn_bytes", w["attn_bytes"]) + w["append_bytes"]
    flush = touched < 4 * l2 or shared_bt is not None   # (shared pages would stay in L2 between steps)
    flush_buf = torch.empty(2 * l2 // 4, dtype=torch.int32, device=dev) if flush else None

    def timed(fn, k_steps, events_per_step=0):
        """k_steps calls of fn on the device; with a flush, each between a flush and its own event
        pair.  Returns (ms per step, per-step marks for events_per_step > 0)."""
        marks = [[torch.cuda.Event(enable_timing=True) for _ in range(events_per_step)] for _ in range(k_steps)]
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(k_steps if flush else 1)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        if not flush:
            pairs[0][0].record(stream)
        for k in range(k_steps):
            if flush:
                flush_buf.fill_(k)
                pairs[k][0].record(stream)
            fn(marks[k])
            if flush:
                pairs[k][1].record(stream)
        if not flush:
            pairs[0][1].record(stream)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in pairs) / k_steps
        return ms, marks

    # ---- device-timed region: exactly K steps, inputs resident in HBM, two events per step (or per run) ----
    nv = NvmlClocks(dev).start()
    time.sleep(0.05)
    w0 = time.perf_counter()
    ms_step, _ = timed(lambda m: step(), args.steps)
    w1 = time.perf_counter()
    time.sleep(0.02)
    nv.stop()
    xystep.check(batch)
    ms_per_step = max_over_ranks(ms_step, world, device=dev)
    clocks = nv.summary(w0, w1) or smi.summary(w0, w1)
    if not clocks or not clocks.get("samples"):
        clocks = smi.summary()

    # ---- instrumented pass (not the timed region): append and attention times per step ----
    def marked(m):
        m[0].record(stream)
        append()
        m[1].record(stream)
        attend()
        m[2].record(stream)
    _, marks = timed(marked, args.steps, 3)
    xystep.check(batch)
    append_ms = statistics.mean(m[0].elapsed_time(m[1]) for m in marks)
    attn_ms = statistics.mean(m[1].elapsed_time(m[2]) for m in marks)

    # how evenly the deal spread the work: one traced launch after the timed region
    deal_trace = None
    if not fp8 and not split:
        trace = torch.zeros(pl.num_ctas, 4, dtype=torch.int64, device=dev)
        xy.xy_paged_attention_traced(vals["q"], batch.cu, batch.ctx, batch.block_table, vals["k_pool"],
                                     vals["v_pool"], wl.scale, wl.causal, pl.tasks, pl.merges, pl.num_ctas,
                                     pl.workspace, pl.task_counter if pl.dynamic else None, trace, batch.err, out)
        torch.cuda.synchronize()
        xystep.check(batch)
        deal_trace = xy.trace_summary(trace.cpu().numpy())
        if wl.num_tokens == wl.num_seqs and wl.group <= 16 and pl.dynamic:
            # the timed launches of a pure decode batch run two half-size CTAs per SM slot; a
            # traced launch keeps one CTA (one record) per slot
            deal_trace["kernel"] = "one decode-path CTA per SM slot (the timed launches run two)"

    value = job_throughput(config, w, ms_per_step / 1e3, world)
    unit, bound = unit_of(config)
    traffic_key = (config + ("_fp8" if fp8 else "") +
                   (f"_s{args.schedule}" if args.schedule != args.default_schedule else ""))
    kname = (attention_kernel(wl, args.kv, args.schedule) if not split else
             "dequant_pages_kernel + meta_attention_kernel + paged_attention_kernel<fp8>")
    attn_s = attn_ms / 1e3
    if bound == "hbm":
        # prefix sharing: the bytes DRAM must deliver are the distinct pages' (the logical bytes,
        # as if every row had its own copy, are reported beside them)
        alg = w.get("unique_attn_bytes", w["attn_bytes"])
        achieved = alg / attn_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s", "frac": achieved / pk["hbm"],
                "traffic": measured_traffic(traffic_key), "kernel": kname, "algorithmic_bytes": alg,
                "avg_launch_ms": attn_ms, "peak_source": pk["source"]}
        if "unique_attn_bytes" in w:
            roof.update({"logical_bytes": w["attn_bytes"], "logical_gbs": w["attn_bytes"] / attn_s / 1e9})
        if config in ("mixed", "verify"):
            # both bounds matter: time at the roofline = bytes / HBM + flops / tensor (the sum, as the
            # two phases need not overlap) and max(.) (perfect overlap)
            t_sum = w["attn_bytes"] / (pk["hbm"] * 1e9) + w["flops"] / (pk["tc"] * 1e12)
            t_max = max(w["attn_bytes"] / (pk["hbm"] * 1e9), w["flops"] / (pk["tc"] * 1e12))
            roof.update({"tensor_achieved_tflops": w["flops"] / attn_s / 1e12, "algorithmic_flops": w["flops"],
                         "combined_frac_sum": t_sum / attn_s, "combined_frac_max": t_max / attn_s})
    else:
        achieved = w["flops"] / attn_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["tc"], "unit": "TFLOP/s",
                "frac": achieved / pk["tc"], "traffic": measured_traffic(traffic_key), "kernel": kname,
                "algorithmic_flops": w["flops"], "avg_launch_ms": attn_ms, "peak_source": pk["source"],
                "frac_of_sustained": achieved / pk["tc_sustained"] if pk.get("tc_sustained") else None}
    roof["frac_nominal"] = (roof["achieved"] / (NOMINAL["hbm"] if roof["bound"] == "hbm" else NOMINAL["tc"]))
    roof["peak_nominal"] = NOMINAL["hbm"] if roof["bound"] == "hbm" else NOMINAL["tc"]
    roof["timed"] = ("attention call (kernel" + (" + combine" if n_merges else "") + "), CUDA events, instrumented "
                     "pass after the timed steps" if not split else
                     "page dequantization + tile attention + 8-bit decode attention (+ combines), CUDA events")
    append_gbs = w["append_bytes"] / (append_ms / 1e3) / 1e9
    append_roof = {"achieved": append_gbs, "unit": "GB/s", "peak": pk["hbm"], "frac": append_gbs / pk["hbm"],
                   "algorithmic_bytes": w["append_bytes"], "avg_ms": append_ms,
                   "timed": "slot mapping + KV append (one fused kernel), CUDA events",
                   "kernel": "kv_append_paged_fp8_kernel" if fp8 else "kv_append_paged_kernel"}

    # ---- end to end through the public API: pinned host inputs in, output out, every step ----
    host = {k: vals[k].cpu().pin_memory() for k in ("q", "k_new", "v_new")}
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    meta = dict(cu=wl.cu_seqlens_q, ctx=wl.context_lens, free=wl.free_list)
    # a serving loop re-plans every step: block table, task table and their upload (packed into
    # one copy by the Planner, created once like an engine's state).  The next step's plan depends
    # only on its lengths, so it is built on the host while this step runs on the device (as an
    # engine's scheduler overlaps the next batch with the current one); every step's timed region
    # holds one plan, its inputs' upload, the step and its output's download.
    planner = xystep.Planner(wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.block_size, wl.max_blocks, wl.causal,
                             device=dev, num_ctas=pl.num_ctas, kv_fp8=fp8, schedule=args.schedule)
    split_planner = (xystep.Fp8SplitPlanner(wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.block_size,
                                            wl.max_blocks, wl.causal, device=dev, num_ctas=pl.num_ctas)
                     if split else None)

    def make_batch(stream=None):
        if split:
            return split_planner.plan(meta["cu"], meta["ctx"], meta["free"], stream=stream)
        return planner.plan(meta["cu"], meta["ctx"], meta["free"], stream=stream, block_table=shared_bt)

    plan_times = []
    out_hosts = [out_host, torch.empty(out.shape, dtype=out.dtype).pin_memory()]
    # inputs go up on one copy stream and outputs come down on another, so that the copy engines
    # overlap the neighbouring steps' kernels (and each other); two device input buffers and two
    # pinned output buffers alternate between steps
    cs_up, cs_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dev_in = [{x: torch.empty_like(vals[x]) for x in ("q", "k_new", "v_new")} for _ in range(2)]
    up_ev = [torch.cuda.Event() for _ in range(2)]      # step k's inputs are on the device
    step_ev = [torch.cuda.Event() for _ in range(2)]    # step k's kernels are done
    down_ev = [torch.cuda.Event() for _ in range(2)]    # step k's output is in host memory
    planner_now = split_planner if split else planner

    def upload(k):
        """Step k's inputs and its freshly planned tables go up on the upload stream (after step k - 2,
        which used the same input and table buffers, is done).  Returns step k's batch."""
        with torch.cuda.stream(cs_up):
            if k >= 2:
                cs_up.wait_event(step_ev[k % 2])
            for x in ("q", "k_new", "v_new"):
                dev_in[k % 2][x].copy_(host[x], non_blocking=True)
        planner_now.wait_upload()   # (the planner's own wait, kept out of the planning time)
        tp = time.perf_counter()
        b = make_batch(stream=cs_up)
        plan_times.append(time.perf_counter() - tp)
        up_ev[k % 2].record(cs_up)
        return b

    def launch(k, b):
        """Step k through the public API on the compute stream, once its inputs and tables are up;
        its output then comes down on the download stream."""
        stream.wait_event(up_ev[k % 2])
        d = dev_in[k % 2]
        if split:
            o = xystep.run_step_fp8_split(b, d["q"], d["k_new"], d["v_new"], vals["k_codes"], vals["v_codes"],
                                          vals["k_scales"], vals["v_scales"], wl.scale)
        elif fp8:
            o = planner.run(b, d["q"], d["k_new"], d["v_new"], vals["k_codes"], vals["v_codes"], wl.scale,
                            k_scales=vals["k_scales"], v_scales=vals["v_scales"])
        else:
            o = planner.run(b, d["q"], d["k_new"], d["v_new"], vals["k_pool"], vals["v_pool"], wl.scale)
        step_ev[k % 2].record(stream)
        with torch.cuda.stream(cs_down):
            cs_down.wait_event(step_ev[k % 2])
            o.record_stream(cs_down)
            out_hosts[k % 2].copy_(o, non_blocking=True)
            down_ev[k % 2].record(cs_down)

    # As a serving loop runs: step k + 1's inputs and tables (planned on the host meanwhile) go up
    # while step k computes, step k's output comes down while step k + 1 computes, and the host
    # waits for step k - 1's output only after step k is enqueued (so the GPU waits neither on the
    # host nor on a copy, and every step's result reaches the host).
    total = args.warmup + args.steps
    t_start = None
    b_next = upload(0)
    for k in range(total):
        if k == args.warmup:
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            t_start = time.perf_counter()
            b_next = upload(k)   # the first timed step's inputs and tables go up inside the timed region
        b_cur = b_next
        launch(k, b_cur)
        if k + 1 < total and k + 1 != args.warmup:
            b_next = upload(k + 1)
        if k >= 1:
            down_ev[(k - 1) % 2].synchronize()   # step k - 1's output is on the host
    down_ev[(total - 1) % 2].synchronize()
    e2e_total = time.perf_counter() - t_start
    h2d = sum(host[x].numel() * 2 for x in host) + planner_now.last_upload_bytes
    d2h = out_host.numel() * 2
    e2e_s = max_over_ranks(e2e_total / args.steps, world, device=dev)
    e2e_val = job_throughput(config, w, e2e_s, world)

    # the task-table build alone (host, into preallocated record arrays), as a step re-plans it
    tt_us = None
    if not split:
        cap_t = np.zeros((int(pl.tasks.shape[0]) + 8, 8), np.int32)
        cap_m = np.zeros((max(1, int(pl.merges.shape[0])) + 8, 8), np.int32)
        tt = []
        for _ in range(25):
            t0 = time.perf_counter()
            xy.xy_build_task_table(wl.cu_seqlens_q, wl.context_lens, wl.num_heads_q, wl.num_heads_kv, wl.head_dim,
                                   wl.causal, pl.num_ctas, pl.q_tile, pl.kv_chunk, pl.schedule, tasks_out=cap_t,
                                   merges_out=cap_m)
            tt.append(time.perf_counter() - t0)
        tt_us = 1e6 * statistics.median(tt[5:])

    cpu = None
    if rank == 0 and world == 1 and cpu_budget > 0:
        secs, sw, desc, seqs, seq_secs = oracle_sample(wl, vals, budget_s=cpu_budget, kv=args.kv)
        cpu = {"value": throughput(config, sw, secs), "unit": unit, "cores": 1, "kind": "oracle",
               "sample": desc + (" (pages not shared: the oracle reads each sequence's own pages)"
                                 if shared_bt is not None else "")}
        # the same sample on every host core (one single-threaded process per core)
        sub, secs_all, ncores, desc_all = oracle_sample_cores(wl, vals, seqs, seq_secs, kv=args.kv)
        cpu["all_cores"] = {"value": throughput(config, work(sub, args.kv), secs_all), "unit": unit,
                            "cores": ncores, "kind": "oracle", "sample": desc_all}

    n_launch_per_step = 1 + sum(1 + (1 if x.merges.shape[0] else 0) for x in parts) + (1 if split and batch.tile
                                                                                      else 0)
    res = {
        "workload": describe(config, args), "value": value, "unit": unit, "ms_per_step": ms_per_step,
        "steps": args.steps, "warmup": args.warmup,
        "tokens_per_s": wl.num_tokens * world / (ms_per_step / 1e3),
        "tflops": w["flops"] / (ms_per_step / 1e3) / 1e12,
        "l2": (f"L2 flushed before every timed step (a {2 * l2 / 1e6:.0f} MB write outside the step's events): the "
               f"step touches {touched / 1e6:.0f} MB" if flush else
               f"no flush: the step touches {touched / 1e6:.0f} MB, far more than the {l2 / 1e6:.0f} MB L2"),
        "step": "kv_append (slot mapping fused) + paged_attention" + (" + combine" if n_merges else "") +
                (" (8-bit pages: tile part on bf16 page copies, decode part on codes)" if split else ""),
        "num_tasks": n_tasks, "num_merges": n_merges, "num_ctas": pl.num_ctas, "schedule": args.schedule,
        "balance" if args.schedule != 4 else "balance_if_dealt": pl.stats["balance"],
        "deal_trace": deal_trace,
        "roofline": roof,
        "append": append_roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3,
                "loop": "per step: inputs H2D from pinned memory (upload stream), tables re-planned on the host "
                        "and uploaded, the step (compute stream), output D2H into pinned memory (download stream); "
                        "step k+1's inputs go up while step k computes, and the host waits for step k's output "
                        "after enqueuing step k+1",
                "plan_us": 1e6 * statistics.median(plan_times[args.warmup:]),
                "task_table_us": tt_us},
        "gpu_launches": n_launch_per_step * args.steps,
        "clocks": clocks,
    }
    del vals, batch, out, host, out_hosts, dev_in, planner, split_planner, flush_buf
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="decode", choices=[c for c in workloads.CONFIGS if c != "tiny"],
                    help="headline batch")
    ap.add_argument("--only", action="store_true", help="measure the headline batch alone")
    ap.add_argument("--impl", default="xy", choices=["xy", "reference"])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"], help="page format of the KV cache")
    ap.add_argument("--schedule", type=int, default=None, choices=[0, 1, 2, 3, 4],
                    help="task-table schedule (default: 4, the dynamic deal)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=4.0, help="seconds of oracle work per reference step")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    args.default_schedule = 4
    if args.schedule is None:
        args.schedule = args.default_schedule

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "xy" else "gloo")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    from paged_kv_varlen_xy_gb300 import build as xybuild
    xybuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk = peaks()
    secondary = {} if args.only else {k: (c, kv) for k, (c, kv) in
                                      (SECONDARY_FP8 if args.kv == "fp8" else SECONDARY).items()
                                      if (c, kv) != (args.config, args.kv)}
    with SmiClocks(dev) as smi:
        head = measure(args.config, args, dev, pk, world, rank, 0 if args.no_cpu_baseline else 12.0, smi)
        extra = {key: measure(c, argparse.Namespace(**{**vars(args), "kv": kv}), dev, pk, world, rank,
                              0 if args.no_cpu_baseline else 5.0, smi)
                 for key, (c, kv) in secondary.items()}
        run_clocks = smi.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3 KV, f16 MMA" if args.kv == "fp8" else "bf16", "data": "synthetic",
            "config": {"workload": head["workload"], "parallelism": f"replicas x{world}", "l2": head["l2"],
                       "step": head["step"], "tokens_per_s": head["tokens_per_s"], "tflops": head["tflops"],
                       "num_tasks": head["num_tasks"], "num_merges": head["num_merges"], "num_ctas": head["num_ctas"],
                       "schedule": head["schedule"], "deal_trace": head["deal_trace"],
                       "also_measured": {k: describe(c, argparse.Namespace(**{**vars(args), "kv": kv}))
                                         for k, (c, kv) in secondary.items()}},
            "roofline": head["roofline"],
            "append": head["append"],
            "cpu_baseline": head["cpu_baseline"],
            "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"],
            "clocks_whole_run": run_clocks,
        }
        line.update(extra)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
