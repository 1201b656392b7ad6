"""Benchmark of the paged KV-cache attention hot path on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference]

A step is one pass of the hot path over one batch: kv_store of the step's new
tokens, then attention over the paged cache.  The headline step is the decode
batch (64 sequences, contexts U[128, 2048], 16 q / 8 kv heads, D=128, a
1024-block pool): value = algorithmic HBM bytes (valid-context K/V + q + out +
the store's rows) / step time.  The same line carries the prefill (varlen
causal, TFLOP/s), long skewed decode and prefix-cached prefill workloads, the
decode kernel's roofline, an end-to-end number through host buffers, clocks,
and the CPU oracle's speed on this host.

Caches rotate over several copies so that consecutive steps never find their
working set in L2 (each copy is larger than the 129 MB L2 or the rotation
spans well over it).

--impl reference times the fp64 CPU oracle (the only other implementation of
the path) on this host on a bounded sample of the same workload.
"""
import os

# The CPU oracle runs one BLAS thread per worker process (the workers are
# spawned and read these when numpy loads).
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import math
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "paged decode-attn HBM GB/s (% of peak); prefill attn TFLOP/s (% of peak)"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in PEAKS_FALLBACK}, "measured"
    except Exception:
        return dict(PEAKS_FALLBACK), "fallback"


# ------------------------------------------------------------ work counting

def decode_bytes(b):
    """Algorithmic bytes of decode attention: valid-context K and V, q, out."""
    kv = int(np.sum(b.context_lens.astype(np.int64))) * b.num_kv_heads * b.head_dim * 2 * 2
    qo = 2 * b.num_seqs * b.num_q_heads * b.head_dim * 2
    return kv + qo


def store_bytes(b):
    """kv_store moves each new K and V row in and out once."""
    return int(b.k.shape[0]) * b.num_kv_heads * b.head_dim * 2 * 2 * 2


def dequant_bytes(w):
    """W4A16-G128 dequantisation reads each 4-bit weight and its share of a
    bf16 scale once and writes one bf16."""
    n, k = w.shape
    return n * k // 2 + n * (k // 128) * 2 + n * k * 2


def time_dequant(pkv, w, dev, steps, warmup, copies=4):
    """Mean CUDA-event time (ms) of one dequantisation of `w`, rotating over
    `copies` input/output pairs (each pair larger than a quarter of L2)."""
    import numpy as np
    import torch

    n, k = w.shape
    packed = [torch.from_numpy(w.packed).to(dev) for _ in range(copies)]
    scales = torch.from_numpy(w.scales.view(np.int16)).view(torch.bfloat16).to(dev)
    out = [torch.empty((n, k), dtype=torch.bfloat16, device=dev) for _ in range(copies)]
    for i in range(warmup):
        pkv.w4a16_dequant(out[i % copies], packed[i % copies], scales)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        pkv.w4a16_dequant(out[i % copies], packed[i % copies], scales)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def time_block_manager(pkv, seed=13, n_seqs=1024, block_size=256):
    """Host cost of the block manager: admit n_seqs prompts of U[256, 4096]
    tokens, half of them opening with one shared 1024-token prefix (a system
    prompt), then free them all; returns µs per admission and per free, and
    the fraction of prompt tokens found in shared blocks."""
    import time

    import numpy as np

    rng = np.random.default_rng(seed)
    system = rng.integers(0, 50000, size=1024).astype(np.int32)
    prompts = []
    for i in range(n_seqs):
        t = rng.integers(0, 50000, size=int(rng.integers(256, 4097))).astype(np.int32)
        if i % 2 == 0:
            t[: min(1024, len(t))] = system[: min(1024, len(t))]
        prompts.append(t)
    blocks = sum((len(t) + block_size - 1) // block_size for t in prompts)
    bm = pkv.BlockManager(blocks, block_size)
    t0 = time.perf_counter()
    cached = [bm.allocate(i, t) for i, t in enumerate(prompts)]
    t1 = time.perf_counter()
    for i in range(n_seqs):
        bm.free(i)
    t2 = time.perf_counter()
    tokens = sum(len(t) for t in prompts)
    return {"us_per_admit": (t1 - t0) / n_seqs * 1e6, "us_per_free": (t2 - t1) / n_seqs * 1e6,
            "prompt_tokens_per_s": tokens / (t1 - t0), "shared_token_fraction": sum(cached) / tokens,
            "sample": f"{n_seqs} prompts, U[256, 4096] tokens, half with a shared 1024-token prefix"}


def prefill_flops(b):
    """4*D*Hq per unmasked (query, key) pair."""
    c = b.cached_lens.astype(np.int64)
    n = b.new_lens.astype(np.int64)
    pairs = int(np.sum(n * c + n * (n + 1) // 2))
    return 4 * b.head_dim * b.num_q_heads * pairs


def prefill_bytes(b):
    """q + out + each sequence's K/V read once."""
    kv = int(np.sum(b.context_lens.astype(np.int64))) * b.num_kv_heads * b.head_dim * 2 * 2
    return kv + 2 * int(b.q.shape[0]) * b.num_q_heads * b.head_dim * 2


# ------------------------------------------------------------ multi-rank timing

def job_throughput(total_ms, steps, units_per_step, world, device="cpu"):
    """Whole-job throughput of `world` replicas: the timed region's length is
    the maximum over ranks, and every rank processed `units_per_step` units per
    step.  Returns (ms per step, units per second across the job).  With more
    than one rank this is a collective of the initialised process group."""
    if world > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_step = total_ms / steps
    return ms_step, world * units_per_step / (ms_step * 1e-3)


# ------------------------------------------------------------ ncu counters

def ncu_traffic(*kernels):
    """DRAM bytes per call (read + write, summed over the call's kernels) from
    the committed ncu summary (profiles/counters.json, keyed by kernel, with
    "@workload" when one kernel is recorded on several workloads), or None
    when a record is missing or its kernel's sources changed since the
    counters were taken (source hash recorded beside them)."""
    import hashlib

    try:
        with open(os.path.join(ROOT, "profiles", "counters.json")) as f:
            recs = json.load(f)
        total = 0
        for kernel in kernels:
            rec = recs[kernel]
            h = hashlib.sha256()
            for src in rec["sources"]:
                with open(os.path.join(ROOT, "paged_kv_cache_241_gb300", src), "rb") as g:
                    h.update(g.read())
            if h.hexdigest()[:16] != rec["source_sha256_16"]:
                return None
            total += int(rec["dram_read_bytes"]) + int(rec["dram_write_bytes"])
        return total
    except Exception:
        return None


# The counters records of each workload's call (see profiles/counters.json).
TRAFFIC_KEYS = {
    "decode": ("paged_decode_kernel<128,2,0>", "decode_merge_kernel<128,2,1>"),
    "longdecode": ("paged_decode_kernel<128,4,1>@longdecode", "decode_merge_kernel<128,4,0>@longdecode"),
    "prefill": ("paged_prefill_kernel<128,2,0,0>",),
    "prefix": ("paged_prefill_kernel<128,2,0,1>@prefix",),
    "mixed": ("paged_prefill_kernel<128,2,1,0>@mixed",),
}


# ------------------------------------------------------------ clock sampling

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ GPU arm

def device_batch(b, dev, fill_cache_on_device, seed):
    """Upload a batch; when the cache was not materialised on the host, fill
    the used blocks on the device with seeded N(0,1) bf16 (same distribution)."""
    import torch

    t = {}

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    t["q"] = bf16(b.q)
    t["k"] = bf16(b.k)
    t["v"] = bf16(b.v)
    t["slot_mapping"] = i32(b.slot_mapping)
    t["block_tables"] = i32(b.block_tables)
    t["context_lens"] = i32(b.context_lens)
    t["cu_q"] = i32(b.cu_seqlens_q)
    t["cu_k"] = i32(b.cu_seqlens_k)
    shape = (b.num_blocks, b.block_size, b.num_kv_heads, b.head_dim)
    if b.k_cache is not None:
        t["k_cache"] = bf16(b.k_cache)
        t["v_cache"] = bf16(b.v_cache)
    else:
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        t["k_cache"] = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
        t["v_cache"] = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    return t


def clone_batch(t):
    return {k: v.clone() for k, v in t.items()}


class Arm:
    """Runs one workload's step on the GPU with rotation over cache copies."""

    def __init__(self, pkv, b, dev, copies, fused=None):
        import torch

        self.pkv, self.b, self.dev = pkv, b, dev
        # A decode step stores its tokens inside the decode launch unless asked
        # to time the two calls separately.
        self.fused = (b.kind == "decode") if fused is None else fused
        base = device_batch(b, dev, b.k_cache is None, b.seed)
        self.copies = [base] + [clone_batch(base) for _ in range(copies - 1)]
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.mtb = b.total_blocks_used
        if b.kind == "decode":
            self.ws = [pkv.decode_workspace(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim,
                                            self.mtb, dev) for _ in range(copies)]
            self.out = [torch.empty((b.num_seqs, b.num_q_heads, b.head_dim), dtype=torch.bfloat16,
                                    device=dev) for _ in range(copies)]
        else:
            self.out = [torch.empty((b.q.shape[0], b.num_q_heads, b.head_dim),
                                    dtype=torch.bfloat16, device=dev) for _ in range(copies)]
            self.pws = pkv.prefill_workspace(dev)
        self.max_q = int(b.new_lens.max())
        torch.cuda.synchronize()

    def store(self, i):
        if self.fused:
            return
        t = self.copies[i % len(self.copies)]
        self.pkv.kv_store(t["k"], t["v"], t["k_cache"], t["v_cache"], t["slot_mapping"],
                          self.status)

    def attend(self, i):
        r = i % len(self.copies)
        t = self.copies[r]
        b = self.b
        if b.kind == "decode" and self.fused:
            self.pkv.paged_decode_store_attn(self.out[r], t["q"], t["k"], t["v"],
                                             t["slot_mapping"], t["k_cache"], t["v_cache"],
                                             t["block_tables"], t["context_lens"], b.scale,
                                             self.ws[r], self.mtb, self.status)
        elif b.kind == "decode":
            self.pkv.paged_decode_attn(self.out[r], t["q"], t["k_cache"], t["v_cache"],
                                       t["block_tables"], t["context_lens"], b.scale, self.ws[r],
                                       self.mtb, self.status)
        else:
            self.pkv.paged_prefill_attn(self.out[r], t["q"], t["k_cache"], t["v_cache"],
                                        t["block_tables"], t["cu_q"], t["cu_k"], self.max_q,
                                        b.scale, workspace=self.pws, dev_status=self.status)

    def run(self, steps, warmup):
        """Time `steps` steps; returns (total ms, mean attention-kernel ms, mean store ms).

        The whole-job total comes from a loop with events only around it; the
        per-kernel means from a second loop with events around each call
        (which themselves take time between the launches)."""
        import torch

        stream = torch.cuda.current_stream()
        for i in range(warmup):
            self.store(i)
            self.attend(i)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(steps):
            self.store(i)
            self.attend(i)
        t1.record(stream)
        torch.cuda.synchronize()
        total = t0.elapsed_time(t1)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            e0, e1, e2 = ev[i]
            e0.record(stream)
            self.store(i)
            e1.record(stream)
            self.attend(i)
            e2.record(stream)
        torch.cuda.synchronize()
        store_ms = sum(e0.elapsed_time(e1) for e0, e1, _ in ev) / steps
        attn_ms = sum(e1.elapsed_time(e2) for _, e1, e2 in ev) / steps
        if int(self.status.item()) != 0:
            raise RuntimeError(f"device status {int(self.status.item()):#x} on {self.b.name}")
        return total, attn_ms, store_ms


def e2e_decode(pkv, b, dev, steps, warmup, copies=4):
    """Decode step through host buffers: every step copies the step's inputs
    from pinned host memory (one packed copy), stores + attends, and copies
    the output back, as a serving loop would run it: the inputs of step i+1
    are copied (own stream) while step i computes, and the output of step i
    is read back (another stream) while step i+1 computes; device input and
    output buffers alternate between two sets, and the caches rotate over
    `copies` copies.  The timed loop replays a CUDA graph of eight such steps.  Returns (ms per step, H2D bytes per step, D2H
    bytes per step)."""
    import torch

    t = device_batch(b, dev, b.k_cache is None, b.seed)
    # The caches rotate over `copies` copies, as in the kernel leg, so no step
    # finds the previous step's K/V in L2.
    caches = [(t["k_cache"], t["v_cache"])] + [(t["k_cache"].clone(), t["v_cache"].clone())
                                               for _ in range(copies - 1)]
    names = ("q", "k", "v", "slot_mapping", "block_tables", "context_lens")
    offs, nbytes = {}, 0
    for k in names:  # packed layout, every input 256-byte aligned
        offs[k] = nbytes
        nbytes += (t[k].numel() * t[k].element_size() + 255) // 256 * 256
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    for k in names:
        n = t[k].numel() * t[k].element_size()
        host[offs[k]:offs[k] + n].copy_(t[k].cpu().contiguous().view(-1).view(torch.uint8))
    stage = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]

    def views(buf):
        return {k: buf[offs[k]:offs[k] + t[k].numel() * t[k].element_size()].view(t[k].dtype)
                .view(t[k].shape) for k in names}

    ins = [views(x) for x in stage]
    shape = (b.num_seqs, b.num_q_heads, b.head_dim)
    out = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    out_host = [torch.empty(shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    mtb = b.total_blocks_used
    ws = [pkv.decode_workspace(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim, mtb, dev)
          for _ in range(2)]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    h2d = nbytes
    d2h = out_host[0].numel() * out_host[0].element_size()
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]

    def step(i, first_in_graph=False):
        # (In a captured graph the first use of each buffer set waits for
        # nothing: replays of the graph run one after another on the stream.)
        j = i % 2
        reuse = not (first_in_graph and i < 2)
        with torch.cuda.stream(up):
            if reuse:
                up.wait_event(computed[j])  # the step that last used this input set is done
            stage[j].copy_(host, non_blocking=True)
            copied[j].record(up)
        comp.wait_event(copied[j])
        if reuse:
            comp.wait_event(read[j])  # this output buffer's previous result was read back
        x = ins[j]
        kc, vc = caches[i % copies]
        pkv.paged_decode_store_attn(out[j], x["q"], x["k"], x["v"], x["slot_mapping"],
                                    kc, vc, x["block_tables"],
                                    x["context_lens"], b.scale, ws[j], mtb, status)
        computed[j].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(computed[j])
            out_host[j].copy_(out[j], non_blocking=True)
            read[j].record(down)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    # Eight steps (copies, kernels, read-backs and the streams' ordering) are
    # captured once into a CUDA graph and replayed, as a serving loop replays
    # its decode step: the host then issues one launch per eight steps
    # instead of about ten calls per step.
    per_graph = 8
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(comp)
    with torch.cuda.stream(side):
        cap = torch.cuda.current_stream()
        comp = cap
        with torch.cuda.graph(graph, stream=cap):
            up.wait_stream(cap)
            down.wait_stream(cap)
            for i in range(per_graph):
                step(i, first_in_graph=True)
            cap.wait_stream(up)
            cap.wait_stream(down)
    comp = torch.cuda.current_stream()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // per_graph)
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(comp)
    for _ in range(reps):
        graph.replay()
    e.record(comp)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item()):#x} in the end-to-end leg")
    ms = s.elapsed_time(e) / (reps * per_graph)
    return ms, h2d, d2h


# ------------------------------------------------------------ oracle timing
#
# The CPU baseline is the fp64 oracle as it stands, run on this host's cores:
# the work of a step (the decode batch's sequences, or a sample of a prefill
# batch's query rows) is spread over a pool of worker processes, one BLAS
# thread each.  The pool is started with `spawn` (a process forked after CUDA
# was initialised can hang), and the caches live in shared memory, so the
# workers attach to them instead of receiving copies.

_ORACLE = {}


def _oracle_worker_init(names, shapes, scale):
    from multiprocessing import shared_memory

    segs = [shared_memory.SharedMemory(name=n) for n in names]
    _ORACLE["segs"] = segs  # keeps the mappings alive
    _ORACLE["kc"] = np.ndarray(shapes[0], dtype=np.uint16, buffer=segs[0].buf)
    _ORACLE["vc"] = np.ndarray(shapes[1], dtype=np.uint16, buffer=segs[1].buf)
    _ORACLE["scale"] = scale


def _oracle_decode_task(args):
    import oracle

    q, bt_row, L = args
    return oracle.paged_decode_attn(q, _ORACLE["kc"], _ORACLE["vc"], bt_row[None, :],
                                    np.array([L], np.int32), _ORACLE["scale"])


def _oracle_prefill_task(args):
    import oracle

    q_seq, bt_row, n, len_k, rows = args
    return oracle.paged_prefill_attn(q_seq, _ORACLE["kc"], _ORACLE["vc"], bt_row[None, :],
                                     np.array([0, n], np.int32), np.array([0, len_k], np.int32),
                                     _ORACLE["scale"], rows=rows)


class OraclePool:
    """Worker processes that run the oracle over one batch's caches (which
    have already been through the oracle's kv_store)."""

    def __init__(self, b, kc, vc, workers=None):
        import multiprocessing as mp
        from multiprocessing import shared_memory

        self.workers = workers or max(1, os.cpu_count() or 1)
        self.segs = []
        names, shapes = [], []
        for a in (kc, vc):
            seg = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, dtype=np.uint16, buffer=seg.buf)[...] = a
            self.segs.append(seg)
            names.append(seg.name)
            shapes.append(a.shape)
        self.pool = mp.get_context("spawn").Pool(self.workers, initializer=_oracle_worker_init,
                                                 initargs=(names, shapes, b.scale))
        self.pool.map(abs, range(self.workers))  # every worker up before any timing

    def map(self, fn, tasks):
        return self.pool.map(fn, tasks, chunksize=1)

    def close(self):
        self.pool.close()
        self.pool.join()
        for seg in self.segs:
            seg.close()
            seg.unlink()


def oracle_decode_batch():
    """The decode workload (64 sequences, contexts U[128, 2048], 16 q / 8 kv
    heads, D 128) with its cache materialised on the host in a pool sized to
    the contexts (the full workload's 1024-block pool differs only in unused
    blocks)."""
    full = wl.decode(fill_cache=False)
    return wl.build_batch("decode", "decode", 2, full.cached_lens, full.new_lens,
                          full.num_q_heads, full.num_kv_heads, full.head_dim,
                          num_blocks=full.total_blocks_used)


def oracle_decode_steps(steps, warmup=1, batch=None):
    """Seconds per decode step of the oracle on all host cores: its kv_store of
    the step's 64 new tokens (one call), then its attention for every sequence
    (a pool task per sequence, longest first).  Returns (s/step, batch, workers)."""
    import oracle

    b = batch or oracle_decode_batch()
    kc, vc = oracle.kv_store(b.k_cache, b.v_cache, b.k, b.v, b.slot_mapping)
    pool = OraclePool(b, kc, vc)
    order = np.argsort(-b.context_lens, kind="stable")
    tasks = [(b.q[s:s + 1], b.block_tables[s], int(b.context_lens[s])) for s in order]
    times = []
    try:
        for i in range(warmup + steps):
            t0 = time.perf_counter()
            oracle.kv_store(b.k_cache, b.v_cache, b.k, b.v, b.slot_mapping)
            pool.map(_oracle_decode_task, tasks)
            if i >= warmup:
                times.append(time.perf_counter() - t0)
    finally:
        pool.close()
    return sum(times) / len(times), b, pool.workers


SAMPLED_PREFILL = {
    "prefill": (lambda: wl.prefill(), 32,
                "16 prompts, U[64, 4096] tokens"),
    "prefix": (lambda: wl.prefix(), 4,
               "32 sequences, k*256 cached + U[1, 512] new tokens"),
    "mixed": (lambda: wl.mixed(), 4,
              "48 decode rows + 8 prompt chunks"),
}


def oracle_prefill_sample(name="prefill"):
    """TFLOP/s of the oracle on all host cores over a sample of a prefill-
    kernel workload (varlen prefill, prefix-cached prefill or the mixed step;
    16 q / 8 kv heads, D 128): every `stride`-th query row of every sequence
    and its last row, each sequence's sampled rows one pool task.  Flops
    count the sampled rows' unmasked keys, as for the kernel.  Returns a
    cpu_baseline record."""
    import oracle

    make, stride, what = SAMPLED_PREFILL[name]
    b = make()
    kc, vc = oracle.kv_store(b.k_cache, b.v_cache, b.k, b.v, b.slot_mapping)
    cu_q, cu_k = b.cu_seqlens_q, b.cu_seqlens_k
    tasks, pairs, nrows = [], 0, 0
    for s in range(b.num_seqs):
        q0, q1 = int(cu_q[s]), int(cu_q[s + 1])
        n, len_k = q1 - q0, int(cu_k[s + 1] - cu_k[s])
        if n == 0:
            continue
        rows = np.unique(np.concatenate([np.arange(0, n, stride), [n - 1]]))
        pairs += int(np.sum(len_k - n + rows + 1))
        nrows += len(rows)
        tasks.append((b.q[q0:q1], b.block_tables[s], n, len_k, rows))
    tasks.sort(key=lambda t: -int(np.sum(t[3] - t[2] + t[4] + 1)))
    pool = OraclePool(b, kc, vc)
    try:
        t0 = time.perf_counter()
        pool.map(_oracle_prefill_task, tasks)
        el = time.perf_counter() - t0
    finally:
        pool.close()
    flops = 4 * b.head_dim * b.num_q_heads * pairs
    return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": pool.workers,
            "kind": "oracle", "seconds": el,
            "sample": f"{name}: one query row in {stride} and the last row of each sequence "
                      f"({what}; {nrows} of {b.q.shape[0]} rows, all {b.num_q_heads} heads)"}


# ------------------------------------------------------------ main

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def run_reference(args):
    """The reference arm: the fp64 oracle on this host's cores, timed on the
    decode workload (every step the whole 64-sequence batch), plus its
    prefill throughput on a row sample."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    per, b, workers = oracle_decode_steps(args.steps, warmup=min(args.warmup, 2))
    gbs = (decode_bytes(b) + store_bytes(b)) / per / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "decode: 64 seqs, contexts U[128,2048], 16 q / 8 kv heads, D=128, "
                               "block 256; per step the 64 new tokens' K/V are stored and decode "
                               "attention runs",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": workers, "kind": "oracle",
                         "sample": "the whole decode batch every step (kv_store in one process, "
                                   "attention one sequence per worker task)"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "prefill": {"cpu_baseline": oracle_prefill_sample("prefill")},
        "prefix": {"cpu_baseline": oracle_prefill_sample("prefix")},
        "mixed": {"cpu_baseline": oracle_prefill_sample("mixed")},
    }
    print(json.dumps(line))
    return 0


DEFAULT_COPIES = {"decode": 4, "longdecode": 3, "prefill": 4, "prefix": 8, "mixed": 8}
MAKERS = {"decode": wl.decode, "longdecode": wl.longdecode, "prefill": wl.prefill,
          "prefix": wl.prefix, "mixed": wl.mixed}


def run_single(args, pkv, dev, peaks, peak_src):
    """One workload alone: `steps` timed steps of store + attention (or of
    the W4A16-G128 dequantisation)."""
    if args.workload == "dequant":
        w = wl.dequant()
        ms = time_dequant(pkv, w, dev, args.steps, args.warmup, copies=args.copies or 4)
        gbs = dequant_bytes(w) / (ms * 1e-3) / 1e9
        print(json.dumps({"workload": "dequant", "steps": args.steps, "warmup": args.warmup,
                          "kernel_ms": ms, "metric": "dequant GB/s", "value": gbs, "unit": "GB/s",
                          "frac": gbs / peaks["hbm_gbs"], "bytes": dequant_bytes(w),
                          "peak_source": peak_src}))
        return 0
    b = MAKERS[args.workload](fill_cache=False)
    arm = Arm(pkv, b, dev, copies=args.copies or DEFAULT_COPIES[args.workload],
              fused=False if args.separate_store else None)
    total, am, sm_ = arm.run(args.steps, args.warmup)
    rec = {"workload": args.workload, "steps": args.steps, "warmup": args.warmup,
           "copies": len(arm.copies), "ms_per_step": total / args.steps, "attn_kernel_ms": am,
           "kv_store_ms": sm_, "fused_store": arm.fused, "peak_source": peak_src}
    if b.kind == "decode":
        nbytes = decode_bytes(b) + (store_bytes(b) if arm.fused else 0)
        ach = nbytes / (am * 1e-3) / 1e9
        rec.update(metric="decode GB/s", value=ach, unit="GB/s",
                   frac=ach / peaks["hbm_gbs"], bytes=nbytes)
    else:
        tf = prefill_flops(b) / (am * 1e-3) / 1e12
        rec.update(metric="prefill TFLOP/s", value=tf, unit="TFLOP/s",
                   frac=tf / peaks["bf16_tflops"], flops=prefill_flops(b))
    print(json.dumps(rec))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-main", action="store_true",
                    help="headline decode step only (no other workloads)")
    ap.add_argument("--workload", default="all",
                    choices=["all", "decode", "longdecode", "prefill", "prefix", "mixed", "dequant"],
                    help="run one workload alone (small runs for profiling)")
    ap.add_argument("--separate-store", action="store_true",
                    help="decode: time kv_store and decode as two calls instead of the fused call")
    ap.add_argument("--copies", type=int, default=0,
                    help="rotating cache copies (0 = the default for each workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch

    import paged_kv_cache_241_gb300 as pkv

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as tdist

        tdist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkv.load()
    peaks, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    gpu_index = getattr(props, "uuid", None)
    sampler = ClockSampler(f"GPU-{gpu_index}" if gpu_index else local)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    if args.workload != "all":
        return run_single(args, pkv, dev, peaks, peak_src)

    # ---- headline: decode batch (4 rotating copies of the 1 GiB pool) ----
    b = wl.decode(fill_cache=False)
    arm = Arm(pkv, b, dev, copies=args.copies or 4, fused=False if args.separate_store else None)
    fused = arm.fused
    sampler.start()
    barrier()
    total_ms, attn_ms, store_ms = arm.run(args.steps, args.warmup)
    barrier()
    step_bytes = decode_bytes(b) + store_bytes(b)
    ms_step, per_s = job_throughput(total_ms, args.steps, step_bytes, world, dev)
    value = per_s / 1e9
    # The fused decode launch also moves the step's new K/V rows.
    kernel_bytes = decode_bytes(b) + (store_bytes(b) if fused else 0)
    achieved = kernel_bytes / (attn_ms * 1e-3) / 1e9
    extra = {}
    if not args.only_main:
        # ---- other workloads of the path ----
        sub = max(20, args.steps // 10)
        for name, make, copies, steps in (("longdecode", wl.longdecode, 3, sub),
                                          ("prefill", wl.prefill, 4, sub),
                                          ("prefix", wl.prefix, 8, sub),
                                          ("mixed", wl.mixed, 8, sub)):
            bb = make(fill_cache=False)
            a2 = Arm(pkv, bb, dev, copies=copies)
            tot, am, sm_ = a2.run(steps, args.warmup)
            rec = {"ms_per_step": tot / steps, "attn_kernel_ms": am, "kv_store_ms": sm_}
            if bb.kind == "decode":
                ach = decode_bytes(bb) / (am * 1e-3) / 1e9
                rec["roofline"] = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                                   "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                                   "traffic": ncu_traffic(*TRAFFIC_KEYS[name]),
                                   "bytes_per_launch": decode_bytes(bb)}
            else:
                tf = prefill_flops(bb) / (am * 1e-3) / 1e12
                rec["tflops"] = tf
                # context: each sequence's K/V read once, plus q and out
                rec["hbm_gbs_kv_once"] = prefill_bytes(bb) / (am * 1e-3) / 1e9
                rec["roofline"] = {"bound": "tensor", "achieved": tf,
                                   "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                   "frac": tf / peaks["bf16_tflops"],
                                   "traffic": ncu_traffic(*TRAFFIC_KEYS[name]),
                                   "flops_per_launch": prefill_flops(bb)}
                kvb = store_bytes(bb) / (sm_ * 1e-3) / 1e9
                rec["kv_store"] = {"GB/s": kvb, "frac": kvb / peaks["hbm_gbs"],
                                   "bytes": store_bytes(bb)}
            extra[name] = rec
            del a2
            torch.cuda.empty_cache()
        # W4A16-G128 weight dequantisation (a 4096 x 14336 projection)
        w = wl.dequant()
        dq_ms = time_dequant(pkv, w, dev, max(50, args.steps // 10), args.warmup)
        dq = dequant_bytes(w) / (dq_ms * 1e-3) / 1e9
        extra["block_manager"] = time_block_manager(pkv)
        extra["w4a16_dequant"] = {"kernel_ms": dq_ms, "bytes": dequant_bytes(w),
                                  "roofline": {"bound": "hbm", "achieved": dq,
                                               "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                               "frac": dq / peaks["hbm_gbs"],
                                               "traffic": ncu_traffic("w4a16_dequant_kernel")}}
        torch.cuda.empty_cache()
    clocks = sampler.stop()
    del arm
    torch.cuda.empty_cache()

    # ---- end to end through host buffers ----
    e2e_ms, h2d, d2h = e2e_decode(pkv, b, dev, max(50, args.steps // 10), args.warmup)
    e2e_ms, e2e_per_s = job_throughput(e2e_ms, 1, step_bytes, world, dev)
    e2e_val = e2e_per_s / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode: 64 seqs, contexts U[128,2048], 16 q / 8 kv heads, D=128, "
                               "block 256, 1024-block permuted pool; per step the 64 new tokens' "
                               "K/V are stored and decode attention runs (fused in one launch "
                               "unless --separate-store)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "4 rotating cache copies (4.3 GB) between consecutive steps",
                   "step_bytes": step_bytes},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": ncu_traffic(*TRAFFIC_KEYS["decode"]),
                     "kernel": ("paged_decode_kernel<128,2,0> (kv_store fused) + decode_merge_kernel"
                                "<128,2,1>" if fused else
                                "paged_decode_kernel<128,2,0> + decode_merge_kernel<128,2,1>"),
                     "bytes_per_launch": kernel_bytes, "peak_source": peak_src,
                     "attn_kernel_ms": attn_ms, "kv_store_ms": store_ms},
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        # split-K decode (+ kv_store when not fused) and the merge, per step
        "gpu_launches": (2 if fused else 3) * args.steps,
        "clocks": clocks,
    }
    line.update(extra)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        steps = 20
        per, sb, workers = oracle_decode_steps(steps)
        line["cpu_baseline"] = {"value": (decode_bytes(sb) + store_bytes(sb)) / per / 1e9,
                                "unit": "GB/s", "cores": workers, "kind": "oracle",
                                "sample": f"the whole 64-sequence decode batch, {steps} steps, "
                                          f"{per:.3f} s per step"}
        for name in SAMPLED_PREFILL:
            if name in line:
                line[name]["cpu_baseline"] = oracle_prefill_sample(name)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
