"""Benchmark of one paged decode step on GB300: the KV append of every sequence's
new token plus decode attention over the paged pool, through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload gqa_batch128|tiny_mha|opt13b_mha|shared_prefix|long_context]

Prints ONE JSON line (rank 0).  A step is one pass of the whole hot path over
the workload's batch: reshape_and_cache (append of the new K/V rows) + decode
attention (plan, partition and merge kernels).  `value` is achieved HBM GB/s of
the step's algorithmic bytes (each sequence's K and V rows once, Q and O once,
the appended rows read and written once) with inputs resident in HBM;
`seq_tokens_per_s` is sum(context_lens) per second.  Under torchrun every rank
runs its own copy of the batch (weak scaling; sequences are independent, no
collective on the data path) and rank 0 reports the max-over-ranks time.

--impl reference times the fp64 CPU oracle on the host cores on bounded samples
of the same workload (the only baseline the pages allow: they ship no code).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_265_gb300 import workload as W  # noqa: E402

METRIC = "paged decode attention: achieved HBM GB/s vs peak; seq-tokens/s per layer"
WORKLOADS = {
    "tiny_mha": 1,
    "opt13b_mha": 2,
    "gqa_batch128": 3,
    "shared_prefix": 4,
    "long_context": 5,
    "gqa_batch32": 6,
    "chunked_prefill": 7,
}
DESCR = {
    1: "tiny_mha_d64: 4 seqs L={1,17,33,100}, MHA 4 heads, d=64, bf16, block 16, 64-block pool, 4-row append",
    2: "opt13b_mha_fp16: 32 seqs L~U[512,2048], MHA 40 heads, d=128, fp16, block 16, 8192-block pool, 32-row append",
    3: "gqa_batch128: 128 seqs L~U[1,4096], GQA 32q/8kv, d=128, bf16, block 16, 40000-block pool, 128-row append",
    4: "shared_prefix_spec5: 64 seqs = 1024-token shared prefix + U[16,512], 5 query rows causal, GQA 32q/8kv, "
       "d=128, bf16, 4096-block pool, 320-row append",
    5: "long_context_skewed: 16 seqs L~U[16384,32768] + 240 seqs L~U[64,1024], GQA 64q/8kv, d=128, bf16, "
       "65536-block pool, 256-row append",
    6: "gqa_batch32 (profiling size): 32 seqs L~U[1,4096], GQA 32q/8kv, d=128, bf16, block 16, 10000-block pool, "
       "32-row append",
    7: "chunked_prefill_256: 16 seqs, history U[1024,4096] + 256-token chunk (256 causal query rows), GQA 32q/8kv, "
       "d=128, bf16, block 16, 5000-block pool, 4096-row append",
}
L2_BYTES = 129 * 1024 * 1024


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak():
    """Dense bf16 tensor TFLOP/s: the measured cuBLAS burst figure (a kernel timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# Sources that define the decode partition kernel and its launch: a change to any of them
# invalidates DRAM counters taken earlier.
DECODE_SOURCES = ("pa_device.cuh", "pa_internal.h", "pa_kernels.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_265_gb300", "csrc")
    for name in DECODE_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per call of the partition kernel and of the merge kernel (a dict with keys
    "partition" and "merge") from the committed ncu summary, if it was taken on the current
    kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "decode_kernel_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return {"partition": e.get("dram_bytes_per_launch_full"), "merge": e.get("merge_dram_bytes_per_launch")}


class Staging:
    """A step's host inputs packed back to back (256-byte aligned) in one pinned host buffer and
    mirrored in one device buffer; `views` are device tensors of the original shapes and dtypes,
    and upload() moves all of them with a single asynchronous copy."""

    def __init__(self, tensors, dev):
        import torch

        offs, off = [], 0
        for t in tensors:
            off = (off + 255) // 256 * 256
            offs.append(off)
            off += t.numel() * t.element_size()
        self.nbytes = off
        self.host = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(off, dtype=torch.uint8, device=dev)
        self.views = []
        for t, o in zip(tensors, offs):
            n = t.numel() * t.element_size()
            self.host[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
            self.views.append(self.dev[o:o + n].view(t.dtype).view(t.shape))
        self.dev.copy_(self.host)

    def upload(self):
        self.dev.copy_(self.host, non_blocking=True)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None
        self.first = ""
        self.t0 = self.t1 = None  # host wall clock at the timed region's start and end

    def region_start(self):
        import datetime

        self.t0 = datetime.datetime.now()

    def region_end(self):
        import datetime

        self.t1 = datetime.datetime.now()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        self.first = ""
        if self.proc is not None:
            # Start the timed region only once nvidia-smi delivers samples: its start-up competes
            # for the CPU that launches the (short) steps.
            import select

            ready, _, _ = select.select([self.proc.stdout], [], [], 5.0)
            if ready:
                self.first = self.proc.stdout.readline()
        time.sleep(0.1)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        self.out = (self.first or "") + (self.out or "")
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        import datetime

        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        sm, smax, inside, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
            ts = None
            if len(r) > 9:
                try:
                    ts = datetime.datetime.strptime(r[9].strip(), "%Y/%m/%d %H:%M:%S.%f")
                except ValueError:
                    ts = None
            inside.append(ts is not None and self.t0 is not None and self.t1 is not None and
                          self.t0 <= ts <= self.t1)
        busy = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        # Prefer the samples taken inside the timed region when there are any; the reasons are
        # collected over every sample, just before and after included.
        busy_in = [s for s, i in zip(sm, inside) if i and smax and s > 0.5 * max(smax)]
        use = busy_in or busy
        return {"sm_mhz": statistics.median(use) if use else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "samples_in_region": sum(inside) if self.t0 is not None else None}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle timing

def oracle_time(w: W.Workload, seq_idx: np.ndarray, threads: int, pools=None):
    """One oracle step (append + attention) over the chosen sequences; returns (seconds, bytes, seq_tokens)."""
    import oracle

    orc = oracle.load()
    kc, vc = pools if pools is not None else (w.key_cache.copy(), w.value_cache.copy())
    per_seq = w.num_new_tokens // max(1, w.num_seqs)      # new rows are grouped by sequence, in order
    rows = (np.asarray(seq_idx)[:, None] * per_seq + np.arange(per_seq)[None, :]).ravel()
    sub = W.Workload(**{**w.__dict__, "context_lens": w.context_lens[seq_idx], "block_tables": w.block_tables[seq_idx],
                        "query": np.ascontiguousarray(w.query[seq_idx]),
                        "new_key": np.ascontiguousarray(w.new_key[rows]),
                        "new_value": np.ascontiguousarray(w.new_value[rows]),
                        "slot_mapping": np.ascontiguousarray(w.slot_mapping[rows])})
    t0 = time.perf_counter()
    orc.reshape_and_cache(sub.new_key, sub.new_value, kc, vc, sub.slot_mapping)
    _, bad = orc.decode_attention(sub.query, kc, vc, sub.block_tables, sub.context_lens, sub.scale, sub.dtype,
                                  num_threads=threads)
    dt = time.perf_counter() - t0
    assert bad == 0
    nbytes = W.attention_bytes(sub) + W.append_bytes(sub)
    return dt, nbytes, int(sub.context_lens.astype(np.int64).sum())


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    import subprocess

    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def cpu_baseline(w: W.Workload, budget_s: float = 12.0, single_s: float = 3.0):
    """The oracle as it stands on all host cores, on a bounded sample of the workload; plus the
    same oracle on one core over a smaller sample."""
    import oracle

    threads = oracle.load().max_threads()
    pools = (w.key_cache.copy(), w.value_cache.copy())
    n = w.num_seqs
    # grow the sample (whole sequences, in batch order) until it takes >= 1 s, then repeat to fill the budget
    k = max(1, min(n, 8))
    while True:
        dt, nbytes, toks = oracle_time(w, np.arange(k), threads, pools)
        if dt >= 1.0 or k == n:
            break
        k = min(n, k * 2)
    reps, tot_t, tot_b, tot_tok = 1, dt, nbytes, toks
    while tot_t < budget_s:
        dt, nbytes, toks = oracle_time(w, np.arange(k), threads, pools)
        reps += 1
        tot_t += dt
        tot_b += nbytes
        tot_tok += toks
    # one core: whole sequences in batch order (cycling) until single_s seconds are spent
    k1, t1, b1, tok1 = 0, 0.0, 0, 0
    while t1 < single_s:
        i = k1 % n
        dt, nbytes, toks = oracle_time(w, np.arange(i, i + 1), 1, pools)
        k1 += 1
        t1 += dt
        b1 += nbytes
        tok1 += toks
    return {"value": tot_b / tot_t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "seq_tokens_per_s": tot_tok / tot_t, "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "sample": f"first {k} of {n} sequences (append + attention), {reps} repetitions, {tot_t:.1f} s",
            "single_core": {"value": b1 / t1 / 1e9, "unit": "GB/s", "seq_tokens_per_s": tok1 / t1,
                            "sample": f"{k1} sequence runs in batch order, {t1:.1f} s"}}


def run_reference(args, rank, world):
    if rank != 0:
        return
    cfg = WORKLOADS[args.workload]
    w = W.WORKLOADS[cfg]()
    import oracle

    threads = oracle.load().max_threads()
    pools = (w.key_cache.copy(), w.value_cache.copy())
    # size each step's sample so warmup + steps fit in about two minutes
    per_step = 120.0 / max(1, args.steps + args.warmup)
    order = np.arange(w.num_seqs)
    dt1, _, _ = oracle_time(w, order[:1], threads, pools)
    k = int(max(1, min(w.num_seqs, per_step / max(dt1, 1e-4))))
    for _ in range(args.warmup):
        oracle_time(w, order[:k], threads, pools)
    tt, tb, ttok = 0.0, 0, 0
    for s in range(args.steps):
        sel = np.roll(order, -s * k)[:k]
        dt, nb, tok = oracle_time(w, np.sort(sel), threads, pools)
        tt += dt
        tb += nb
        ttok += tok
    value = tb / tt / 1e9
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": DESCR[cfg], "sample_seqs_per_step": k},
            "seq_tokens_per_s": ttok / tt,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{k} of {w.num_seqs} sequences per step (append + attention)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def run_ours(args, rank, world, local):
    import torch

    from paged_kv_cache_265_gb300 import build as B
    from paged_kv_cache_265_gb300 import pa

    if rank == 0 or world == 1:
        B.build()
    barrier(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = WORKLOADS[args.workload]
    w = W.WORKLOADS[cfg]()
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[w.dtype]

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(tdt)

    kc, vc = up(w.key_cache), up(w.value_cache)
    kv8 = args.kv == "fp8"
    K_SCALE, V_SCALE = 0.05, 0.03
    if kv8:   # the same history, quantised to FP8 E4M3 with one scale per cache
        kc = (kc.float() / K_SCALE).to(torch.float8_e4m3fn).view(torch.uint8)
        vc = (vc.float() / V_SCALE).to(torch.float8_e4m3fn).view(torch.uint8)
        torch.cuda.empty_cache()
    # A step's inputs live back to back in one device buffer (views below), mirrored by one
    # pinned host buffer, so the end-to-end loop uploads them with a single copy per step.
    host_in = [torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(tdt)
               for x in (w.query, w.new_key, w.new_value)]
    host_in += [torch.from_numpy(x) for x in (w.slot_mapping, w.block_tables, w.context_lens)]
    staging = Staging(host_in, dev)
    q, nk, nv, sm, bt, cl = staging.views
    out = torch.empty_like(q)
    # A batch whose sequences share prefix blocks declares them as one prefix group (as the
    # block manager that mapped them would); the prefix is then attended once per kv head.
    groups = None
    if w.shared_prefix_blocks and not kv8 and not args.no_prefix_groups:
        groups = ([0, w.num_seqs], [w.shared_prefix_blocks * w.block_size])
        ws = pa.alloc_workspace_shared_prefix(w.num_seqs, w.q_len, w.num_heads, w.head_dim, w.max_context_len,
                                              args.partition, device=dev)
    else:
        ws = pa.alloc_workspace(w.num_seqs, w.q_len, w.num_heads, w.head_dim, w.max_context_len, args.partition,
                                device=dev)
    pa.set_decode_math(args.math)
    stream = torch.cuda.current_stream(dev)
    pa.get_device_error(clear=True)

    def step(inputs=None, o=None):
        q_, nk_, nv_, sm_, bt_, cl_ = inputs if inputs is not None else (q, nk, nv, sm, bt, cl)
        o = out if o is None else o
        if kv8:
            pa.reshape_and_cache_fp8(nk_, nv_, kc, vc, sm_, K_SCALE, V_SCALE, stream=stream)
            n1 = pa.last_launch_count()
            pa.decode_attention_fp8kv(o, q_, kc, vc, bt_, cl_, w.scale, w.max_context_len, ws, K_SCALE, V_SCALE,
                                      partition_size=args.partition, stream=stream)
            return n1 + pa.last_launch_count()
        pa.reshape_and_cache(nk_, nv_, kc, vc, sm_, stream=stream)
        n1 = pa.last_launch_count()
        if groups:
            pa.decode_attention_shared_prefix(o, q_, kc, vc, bt_, cl_, w.scale, w.max_context_len, ws, *groups,
                                              partition_size=args.partition, stream=stream)
        else:
            pa.decode_attention(o, q_, kc, vc, bt_, cl_, w.scale, w.max_context_len, ws,
                                partition_size=args.partition, stream=stream)
        return n1 + pa.last_launch_count()

    attn_bytes = W.attention_bytes(w, 1 if kv8 else None)
    unique_bytes = W.unique_attention_bytes(w, 1 if kv8 else None)  # shared blocks counted once
    step_bytes = attn_bytes + W.append_bytes(w, 1 if kv8 else None)
    seq_tokens = int(w.context_lens.astype(np.int64).sum())
    flush = None
    if step_bytes < 2 * L2_BYTES:   # small working set: flush L2 between steps
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    # --- device-resident timed region (the hot path exactly as a caller runs it).  Each L2 flush
    # is bracketed by its own event pair and its time taken out (a flush costs differently when
    # it runs between steps than when flushes run back to back).
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def flushed():
        """Runs the L2 flush; returns its (start, stop) events when timed."""
        if flush is None:
            return None
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        flush.zero_()
        b.record(stream)
        return a, b

    flush_events = []
    with ClockSampler(local) as clocks:
        # The warm-up steps run here, after the clock sampler has started, so that the GPU goes
        # from them straight into the timed region instead of idling through the sampler's start.
        for _ in range(max(3, args.warmup)):
            ev = flushed()
            launches_per_step = step()
        partition_used = pa.last_partition_size()
        barrier(world)
        torch.cuda.synchronize(dev)
        clocks.region_start()
        start.record(stream)
        for _ in range(args.steps):
            ev = flushed()
            if ev:
                flush_events.append(ev)
            step()
        stop.record(stream)
        torch.cuda.synchronize(dev)
        clocks.region_end()
        barrier(world)
    total_ms = start.elapsed_time(stop)
    flush_ms = sum(a.elapsed_time(b) for a, b in flush_events)
    step_ms_local = max(1e-9, (total_ms - flush_ms) / args.steps)
    step_ms = max_over_ranks(step_ms_local, world, dev)

    # --- kernel times for the roofline: the same steps again, with the library's CUDA events
    # recorded on the launch stream around the plan, partition and merge kernels of every call.
    # (Events between launches suspend the programmatic overlap of launch set-up, which is
    # why the step itself is timed without them.)
    # Pass 1 times the partition and merge kernels as one span (their programmatic overlap kept):
    # the roofline figure.  Pass 2 times the plan, partition and merge kernels apart.
    prof_steps = min(args.steps, 2048)
    spans = []
    for mode in (2, 1):
        pa.profile_enable(mode)
        pa.profile_read_parts()
        for _ in range(prof_steps):
            flushed()
            step()
        torch.cuda.synchronize(dev)
        spans.append(pa.profile_read_parts())
    pa.profile_enable(False)
    _, attn_ms_total, _, attn_n = spans[0]
    plan_ms_total, kern_ms_total, merge_ms_total, kern_n = spans[1]
    err = pa.get_device_error(clear=True)

    # --- the append alone (the KV-append kernel), timed over the same number of calls
    ap_n = max(1, min(args.steps, 500))
    ap_s, ap_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    ap_s.record(stream)
    for _ in range(ap_n):
        if kv8:
            pa.reshape_and_cache_fp8(nk, nv, kc, vc, sm, K_SCALE, V_SCALE, stream=stream)
        else:
            pa.reshape_and_cache(nk, nv, kc, vc, sm, stream=stream)
    ap_e.record(stream)
    torch.cuda.synchronize(dev)
    append_ms = ap_s.elapsed_time(ap_e) / ap_n
    append_bytes = W.append_bytes(w, 1 if kv8 else None)

    # --- end to end through the public API: host inputs in, host output back, every step
    # (query, new K/V rows, slot mapping, block tables and context lengths in one pinned buffer).
    # As a serving loop would, a copy stream uploads step i + 1's inputs into the second of two
    # device buffers and downloads step i's output while step i computes.
    stagings = [staging, Staging(host_in, dev)]
    outs = [out, torch.empty_like(out)]
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = staging.nbytes
    d2h = h_out.numel() * h_out.element_size()
    e2e_steps = max(1, min(args.steps, 200))
    copy_stream = torch.cuda.Stream(dev)

    def e2e_run(n):
        ev_up = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        with torch.cuda.stream(copy_stream):
            stagings[0].upload()
            ev_up[0].record(copy_stream)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                with torch.cuda.stream(copy_stream):
                    if i >= 1:
                        copy_stream.wait_event(ev_done[b ^ 1])  # step i - 1 is done with that buffer
                    stagings[b ^ 1].upload()
                    ev_up[b ^ 1].record(copy_stream)
            stream.wait_event(ev_up[b])
            ev = flushed()
            if ev:
                e2e_flush.append(ev)
            step(stagings[b].views, outs[b])
            ev_done[b].record(stream)
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(ev_done[b])
                h_out.copy_(outs[b], non_blocking=True)
        stream.wait_stream(copy_stream)

    e2e_flush = []
    e2e_run(3)
    torch.cuda.synchronize(dev)
    e2e_flush.clear()
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    es.record(stream)
    copy_stream.wait_event(es)
    e2e_run(e2e_steps)
    ee.record(stream)
    torch.cuda.synchronize(dev)
    e2e_flush_ms = sum(a.elapsed_time(b) for a, b in e2e_flush)
    e2e_ms = max_over_ranks((es.elapsed_time(ee) - e2e_flush_ms) / e2e_steps, world, dev)

    total_bytes = sum_over_ranks(step_bytes, world, dev)
    total_tokens = sum_over_ranks(seq_tokens, world, dev)
    if rank != 0:
        return
    peak, peak_kind = peaks()
    kern_ms = kern_ms_total / max(1, kern_n)          # K2: the partition pass (or the tcgen05 kernel)
    merge_ms = merge_ms_total / max(1, kern_n)        # K3: the log-sum-exp merge (0 without one), timed apart
    plan_ms = plan_ms_total / max(1, kern_n)
    attn_ms = attn_ms_total / max(1, attn_n)          # K2 + K3 as one span, the attention proper
    achieved = attn_bytes / (attn_ms * 1e-3) / 1e9
    achieved_k2 = attn_bytes / (kern_ms * 1e-3) / 1e9
    # The library runs a call with >= 128 query rows per kv head (and the default split) on the
    # tcgen05 prefill kernel, everything else on the split-K decode kernel.
    tc_path = not kv8 and not groups and (args.math == "tcgen05" or
                                          (args.math == "auto" and (w.num_heads // w.num_kv_heads) * w.q_len >= 128))
    # A shared-prefix call with >= 16 query rows per kv head runs wholly on tcgen05: after the
    # order kernel (marks 0-1), the suffix kernel (1-2) then the prefix kernel (2-3), which merges
    # both pieces.
    tc_shared = bool(groups) and not kv8 and (w.num_heads // w.num_kv_heads) * w.q_len >= 16
    kernel_name = ("prefill_tc_kernel (tcgen05, no split)" if tc_path and not groups else
                   "suffix_tc_kernel + prefix_tc_kernel (tcgen05: each sequence's positions after its shared "
                   "prefix, longest first, then each prefix once per kv head for the group's rows, merging both "
                   "pieces)"
                   if tc_shared else
                   "prefix_tc_kernel + decode_kernel + merge_kernel (shared prefix on tcgen05, the rest split-K, "
                   "log-sum-exp merge)" if groups else
                   "decode_kernel + merge_kernel (split-K partition pass and log-sum-exp merge)")
    t = ncu_traffic(args.workload) if not kv8 and not tc_path and args.math == "auto" else None
    traffic = t["partition"] + t["merge"] if t and t["partition"] and t["merge"] is not None else None
    flops = W.attention_flops(w)
    tpeak, tpeak_kind = tensor_peak()
    compute_bound = flops / attn_bytes > tpeak * 1e12 / (peak * 1e9)   # past the ridge point
    line = {
        "metric": METRIC, "value": total_bytes / (step_ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": DESCR[cfg], "seq_tokens_per_step": seq_tokens, "bytes_per_step": step_bytes,
                   "attention_bytes": attn_bytes, "partition_tokens": partition_used or None, "math": args.math,
                   "kv_cache": args.kv, "prefix_groups": len(groups[1]) if groups else 0,
                   "l2": "flushed between steps" if flush is not None else
                   f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB per step vs 129 MB L2)",
                   "parallelism": f"{world} independent replicas" if world > 1 else "1 GPU"},
        "seq_tokens_per_s": total_tokens / (step_ms * 1e-3),
        "query_tokens_per_s": sum_over_ranks(w.num_seqs * w.q_len, world, dev) / (step_ms * 1e-3),
        "unique_attention_bytes": unique_bytes,
        "append": {"us_per_call": append_ms * 1e3, "bytes": append_bytes,
                   "gbs": append_bytes / (append_ms * 1e-3) / 1e9},
        "roofline": ({"bound": "tensor", "achieved": flops / (attn_ms * 1e-3) / 1e12, "peak": tpeak,
                      "unit": "TFLOP/s", "frac": flops / (attn_ms * 1e-3) / 1e12 / tpeak,
                      "peak_source": f"{tpeak_kind} dense bf16 cuBLAS burst", "flops_per_launch": flops,
                      "kernel": kernel_name, "kernel_ms": attn_ms, "traffic": traffic,
                      "hbm_gbs": achieved}
                     if compute_bound else
                     {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                      "frac": achieved / peak, "peak_source": f"{peak_kind} copy bandwidth",
                      "kernel": kernel_name, "kernel_ms": attn_ms,
                      "traffic": traffic, "tflops": flops / (attn_ms * 1e-3) / 1e12,
                      "partition_kernel": {"ms": kern_ms, "achieved": achieved_k2, "frac": achieved_k2 / peak,
                                           "traffic": t["partition"] if t else None},
                      "merge_kernel_ms_apart": merge_ms, "plan_kernel_ms_apart": plan_ms,
                      "part_kernels": ({"partition_kernel": "suffix_tc_kernel", "merge_kernel_ms_apart":
                                        "prefix_tc_kernel", "plan_kernel_ms_apart": "suffix_order_kernel"}
                                       if tc_shared else
                                       {"partition_kernel": "decode_kernel", "merge_kernel_ms_apart":
                                        "merge_kernel", "plan_kernel_ms_apart": "plan_kernel"})}),
        "gpu_launches": launches_per_step * args.steps,
        "roofline_steps": attn_n,
        "clocks": clocks.summary(),
        "device_error_flags": err,
        "e2e": {"value": total_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)


def run_copy_blocks(args, rank, world, local):
    """Copy-on-write block copy on the GQA pool shape: 8192 random (src, dst) pairs per step,
    each moving a 32 KB K block and a 32 KB V block (read + write)."""
    import torch

    from paged_kv_cache_265_gb300 import build as B
    from paged_kv_cache_265_gb300 import pa

    B.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    nb, hkv, d, pairs = 40000, 8, 128, 8192
    kc = torch.randn((nb, 16, hkv, d), device=dev).to(torch.bfloat16)
    vc = torch.randn((nb, 16, hkv, d), device=dev).to(torch.bfloat16)
    g = np.random.Generator(np.random.PCG64(2656))
    perm = g.permutation(nb)
    mapping = torch.from_numpy(np.stack([perm[:pairs], perm[pairs:2 * pairs]], 1).astype(np.int64)).to(dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        pa.copy_blocks(kc, vc, mapping, stream=stream)
    torch.cuda.synchronize(dev)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        s0.record(stream)
        for _ in range(args.steps):
            pa.copy_blocks(kc, vc, mapping, stream=stream)
        s1.record(stream)
        torch.cuda.synchronize(dev)
    ms = s0.elapsed_time(s1) / args.steps
    nbytes = pairs * 2 * (16 * hkv * d * 2) * 2   # K and V blocks, read and written
    peak, kind = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({"metric": "copy-on-write block copy: achieved HBM GB/s", "value": gbs, "unit": "GB/s",
                      "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                      "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                      "config": {"workload": f"{pairs} pairs of 16x{hkv}x{d} bf16 K and V blocks in a {nb}-block pool",
                                 "bytes_per_step": nbytes},
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                                   "peak_source": f"{kind} copy bandwidth"},
                      "clocks": clocks.summary(), "device_error_flags": pa.get_device_error(clear=True)}),
          flush=True)


def run_spec_verify(args, rank, world, local):
    """Speculative-decoding verification on 64 sequences x (4 drafts + 1), vocabulary 32000:
    the accept/reject scan and the final draw, in one launch."""
    import torch

    from paged_kv_cache_265_gb300 import build as B
    from paged_kv_cache_265_gb300 import pa

    B.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    x = W.spec_verify_inputs(num_seqs=64, k=4, vocab=32000)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    tp, dp, dt, ua, us = d(x.target_probs), d(x.draft_probs), d(x.draft_tokens), d(x.u_accept), d(x.u_sample)
    acc = torch.empty(64, dtype=torch.int32, device=dev)
    out = torch.empty((64, 5), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
    for _ in range(max(3, args.warmup)):
        pa.spec_verify(tp, dp, dt, ua, us, acc, out, stream=stream)
    torch.cuda.synchronize(dev)
    # algorithmic bytes: the rows each sequence's draw reads (two at a rejection, one for the bonus)
    na = acc.cpu().numpy()
    rows = sum(2 if a < 4 else 1 for a in na)
    nbytes = rows * 32000 * 4 + 64 * 4 * (8 + 4 + 4) + 64 * 4 * 6
    tot = 0.0
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for _ in range(args.steps):
        flush.zero_()
        ev[0].record(stream)
        pa.spec_verify(tp, dp, dt, ua, us, acc, out, stream=stream)
        ev[1].record(stream)
        torch.cuda.synchronize(dev)
        tot += ev[0].elapsed_time(ev[1])
    ms = tot / args.steps
    # The same timing around a one-element fill, after the same flush: what this method
    # measures for a launch that does almost nothing.
    tiny = torch.empty(1, dtype=torch.int32, device=dev)
    floor = []
    for _ in range(min(args.steps, 200)):
        flush.zero_()
        ev[0].record(stream)
        tiny.fill_(1)
        ev[1].record(stream)
        torch.cuda.synchronize(dev)
        floor.append(ev[0].elapsed_time(ev[1]))
    floor_ms = float(np.median(floor))
    peak, kind = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({"metric": "speculative verification: achieved HBM GB/s", "value": gbs, "unit": "GB/s",
                      "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                      "higher_is_better": True, "dtype": "f32", "data": "synthetic",
                      "config": {"workload": "64 sequences, 4 drafts + 1, vocabulary 32000, L2 flushed per launch",
                                 "bytes_per_step": nbytes, "accepted_histogram": np.bincount(na, minlength=5).tolist(),
                                 "launch_floor_ms": floor_ms},
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                                   "peak_source": f"{kind} copy bandwidth"},
                      "device_error_flags": pa.get_device_error(clear=True)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="gqa_batch128")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--partition", type=int, default=0,
                    help="split-K partition in tokens (a multiple of 16); 0 lets the library choose")
    ap.add_argument("--no-prefix-groups", action="store_true",
                    help="run a shared-prefix batch through the plain multi-query call (no prefix group declared)")
    ap.add_argument("--op", choices=["decode_step", "copy_blocks", "spec_verify"], default="decode_step",
                    help="decode_step: the timed hot path; copy_blocks / spec_verify: those steps alone")
    ap.add_argument("--kv", choices=["16bit", "fp8"], default="16bit",
                    help="KV cache element type: the workload's 16-bit type, or FP8 E4M3 with per-cache scales")
    ap.add_argument("--math", choices=["auto", "fma", "tensor", "tcgen05"], default="auto",
                    help="attention arithmetic (auto: CUDA cores for one row per kv head, mma.sync tiles for "
                         "grouped heads and short chunks, the tcgen05 kernel from 128 rows per kv head)")
    args = ap.parse_args()
    rank, world, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        elif args.op == "copy_blocks":
            run_copy_blocks(args, rank, world, local)
        elif args.op == "spec_verify":
            run_spec_verify(args, rank, world, local)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
