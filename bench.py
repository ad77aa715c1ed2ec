"""Benchmark of the quantized-KV decode hot path on one or more GPUs.

One step = one decode step of the workload (for the paged serving workload:
kvq_append of one new token per sequence, then kvq_decode) over a cache that
is already resident in HBM.  The timed region holds exactly --steps steps,
bracketed by a barrier and a device synchronize; steps rotate over enough
identical cache replicas that the bytes cycled exceed 4x the L2 size (or the
cache alone exceeds L2), so every step reads its cache from HBM.

Prints one JSON line (rank 0): the headline workload (the paged int8 serving
step, the largest single-GPU one) and, at one GPU, a per_config object with the
same measurements for each of the five named workloads (decode roofline,
same-design bf16-cache kernel, and the float64 oracle timed on a bounded sample
on the host cores).  --impl reference times the float64 CPU oracle (the
reference arm) on a bounded sample of the same workload.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The headline: the largest single-GPU workload (paged int8 serving step,
# 2.39 GB of cache per step).  Every named workload is measured too (per_config).
DEFAULT_WORKLOAD = "paged_int8_b64_len2k_32k"
ALL_WORKLOADS = ["int8_b1_h4_t256", "gqa_int8_window128_b8_t4096", "int4_factor_b32_len1k_8k",
                 "paged_int8_b64_len2k_32k", "long_k4v8_b4_t131072"]
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def decode_kernel_hash() -> str:
    """sha256[:12] of the default-path decode sources with comments and blank
    lines removed (editing a comment does not invalidate a recorded capture)."""
    import re
    h = hashlib.sha256()
    for f in ("kvq_decode_impl.cuh", "kvq_decode.cu", "kvq_device.cuh"):  # the default-path kernels
        src = open(os.path.join(ROOT, "quantized_kv_cache_07_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        src = "\n".join(line.rstrip() for line in src.splitlines() if line.strip())
        h.update(src.encode())
    return h.hexdigest()[:12]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary, valid only for the
    decode sources it was captured from (matched by source hash)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    want = decode_kernel_hash()
    for line in open(p):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == workload and parts[1] == kernel \
                and parts[2] == want:
            return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def cache_bytes_per_step(inp) -> int:
    """Algorithmic bytes one decode step reads: codes + scales of every cached
    quantized token and the bf16 window tokens, per KV head."""
    w = inp.workload
    L = inp.decode_lengths.astype(int)
    D = w.head_dim
    if w.k_bits == 2:
        # 2-bit codes of K and V plus one 16-byte metadata record per 16-token block
        lq = [max(int(l) - w.window, 0) if w.window else int(l) for l in L]
        return w.kv_heads * sum(2 * D * 2 // 8 * x + 16 * ((x + 15) // 16) + 4 * D * (int(l) - x)
                                for l, x in zip(L, lq))
    per_q = (D * w.k_bits // 8 + D * w.v_bits // 8
             + (0 if w.k_bits == 16 else (16 if w.asym else 8)) - (4 if w.k_per_channel else 0))
    if w.window:
        lq = [max(int(l) - w.window, 0) for l in L]
        lw = [int(l) - x for l, x in zip(L, lq)]
        return w.kv_heads * (per_q * sum(lq) + 4 * D * sum(lw))
    return w.kv_heads * per_q * int(sum(L))


# Chunked prefill (kvq_prefill): each of `batch` sequences holds a quantized
# prefix and takes a chunk of new positions in one call, which quantizes them
# into the cache and lets each attend causally to its sequence up to itself.
PREFILL = dict(name="prefill_int8_b8_prefix1920_chunk128", batch=8, q_heads=32, kv_heads=8, k_bits=8, v_bits=8,
               prefix=1920, chunk=128)
# Decode calls declare their lengths and block tables ready ahead of the
# previous kernel (KVQ_DECODE_GEOMETRY_READY): every step's tables and lengths
# are written before the timed steps, and the kernels just ahead of a decode
# (the previous step's decode, kvq_append) write queries, outputs and cache
# entries only.
DECODE_FLAGS = 1
# The 2-bit token-group format is timed on the shape of this workload.
INT2_SHAPE = "int4_factor_b32_len1k_8k"


def token_head_bytes(k_bits: int, v_bits: int) -> int:
    """Stored bytes of one token of one KV head in the symmetric 8-/4-bit
    formats: K and V codes plus one fp32 scale each."""
    return 128 * k_bits // 8 + 128 * v_bits // 8 + 8


def prefill_row_bytes(prefix: int, chunk: int, batch: int, kv_heads: int, per_token: int) -> int:
    """Cache bytes the rows of one prefill call read: the row at position p
    attends to positions 0..p of its sequence, for every KV head."""
    return batch * kv_heads * per_token * sum(p + 1 for p in range(prefix, prefix + chunk))


# ------------------------------------------------------------------ reference arm / CPU baseline
CPU_SAMPLE_SNIPPET = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from synth import WORKLOADS, make_inputs
from oracle import kvq_oracle as O
w = WORKLOADS[{name!r}]
if {batch}:
    w = w.with_(batch={batch})
if {bf16}:
    w = w.with_(k_bits=16, v_bits=16, window=0, channel_factor=False)
if {asym}:
    w = w.with_(asym=True)
QBITS = {qbits}
inp = make_inputs(w)
G = w.group
budget = {budget}
rng = np.random.default_rng(5)
units = [(int(b), int(h)) for b in rng.permutation(w.batch) for h in range(w.kv_heads)]
per_tok = (128 * w.k_bits // 8 + 128 * w.v_bits // 8 + (0 if w.k_bits in (16, 2) else (16 if w.asym else 8))
           - (4 if w.k_per_channel else 0))
tot_t, tot_b, n, i = 0.0, 0, 0, 0
while tot_t < budget or n == 0:
    b, h = units[i % len(units)]; i += 1
    a, e = inp.seq_offsets[b], inp.seq_offsets[b + 1]
    k = O.bf16_to_f64(inp.k[a:e, h:h+1]); v = O.bf16_to_f64(inp.v[a:e, h:h+1])
    if w.append_one:
        k = np.concatenate([k, O.bf16_to_f64(inp.k_new[b:b+1, h:h+1])])
        v = np.concatenate([v, O.bf16_to_f64(inp.v_new[b:b+1, h:h+1])])
    c = None if inp.channel_factor is None else inp.channel_factor[h:h+1].astype(np.float64)
    st = O.quantize_sequence(k, v, w.k_bits, w.v_bits, window=w.window, c=c, asym=w.asym,
                             k_per_channel=w.k_per_channel)   # untimed
    t1 = time.perf_counter()
    kh, vh = O.reconstruct_sequence(st, 0)
    qv = O.bf16_to_f64(inp.q[b, h*G:(h+1)*G])
    if QBITS == 8:
        qv = O.effective_query(qv, None if c is None else c[0])
    O.attention(qv, kh, vh)
    tot_t += time.perf_counter() - t1
    L = k.shape[0]; Lq = st["Lq"]
    tot_b += per_tok * Lq + 512 * (L - Lq) + (16 * ((Lq + 15) // 16) if w.k_bits == 2 else 0); n += 1
print(json.dumps({{"seconds": tot_t, "bytes": tot_b, "units": n, "distinct_units": min(n, len(units))}}))
"""

# The oracle runs single-threaded: these variables pin numpy's BLAS to one thread.
CPU_THREAD_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def start_cpu_sample(name: str, budget_s: float, bf16: bool = False, asym: bool = False, qbits: int = 16,
                     batch: int = 0):
    """Start the oracle's decode (dequantize + attention, float64) on a bounded
    sample of the workload's units in a fresh single-threaded process (`batch`:
    the workload with that many sequences instead)."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", **CPU_THREAD_ENV)
    code = CPU_SAMPLE_SNIPPET.format(root=ROOT, name=name, budget=budget_s, bf16=bf16, asym=asym, qbits=qbits,
                                     batch=batch)
    return subprocess.Popen([sys.executable, "-c", code], stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                            env=env)


def finish_cpu_sample(proc, timeout: float = 1800) -> dict:
    out, err = proc.communicate(timeout=timeout)
    if proc.returncode != 0:
        raise RuntimeError("oracle sample failed: " + err[-2000:])
    return json.loads(out.strip().splitlines()[-1])


def run_cpu_sample(name: str, budget_s: float, **kw) -> dict:
    return finish_cpu_sample(start_cpu_sample(name, budget_s, **kw))


def cpu_baseline_entry(d: dict, wname: str) -> dict:
    return {"value": round(d["bytes"] / d["seconds"] / 1e9, 4), "unit": "GB/s", "cores": 1,
            "host_cores": host_cores(), "blas_threads": 1, "kind": "oracle",
            "sample": f"{d['units']} (sequence, kv_head) unit decodes ({d['distinct_units']} distinct) of {wname}, "
                      f"float64 dequantize + attention, one thread (BLAS pinned to 1 thread), "
                      f"{d['seconds']:.1f} s of CPU work on a host with {host_cores()} cores"}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's time (all ranks get the same value)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ GPU arm
class GpuArm:
    """Builds a workload's cache replicas on the device and times its steps."""

    def __init__(self, args, dev, world, local):
        import torch
        from quantized_kv_cache_07_gb300 import _lib
        self.torch, self.lib = torch, _lib
        self.args, self.dev, self.world, self.local = args, dev, world, local
        props = torch.cuda.get_device_properties(dev)
        self.l2 = getattr(props, "L2_cache_size", 0) or 132 * 2 ** 20

    def build_replicas(self, inp_):
        from quantized_kv_cache_07_gb300.cache import cache_for_inputs, fill_from_inputs
        base = cache_for_inputs(inp_, self.dev)
        table, lens = fill_from_inputs(base, inp_, self.dev)
        nbytes = base.allocated_bytes()
        reps = max(1, math.ceil(4 * self.l2 / max(cache_bytes_per_step(inp_), 1)))
        reps = min(reps, 64)
        replicas = [base]
        for _ in range(reps - 1):
            c = cache_for_inputs(inp_, self.dev)
            for name in ("k_codes", "v_codes", "meta", "k_window", "v_window"):
                src, dst = getattr(base, name), getattr(c, name)
                if src is not None:
                    dst.copy_(src)
            replicas.append(c)
        self.torch.cuda.synchronize()
        return replicas, table, lens, nbytes

    def run(self, inp_):
        import numpy as np
        torch, _lib, args, dev, world = self.torch, self.lib, self.args, self.dev, self.world
        import torch.distributed as dist
        from quantized_kv_cache_07_gb300.cache import DecodeWorkspace
        wl = inp_.workload
        replicas, table, lens, alloc = self.build_replicas(inp_)
        B, Hq = wl.batch, wl.q_heads
        q = torch.from_numpy(inp_.q.view(np.int16)).to(dev).view(torch.bfloat16)
        out = torch.empty((B, Hq, 128), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        ws = DecodeWorkspace(replicas[0], B, Hq, args.stream_ctas)
        plan = _lib.kvq_decode_device_plan(replicas[0].desc, B, Hq, args.stream_ctas)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        dec_lens = torch.from_numpy(inp_.decode_lengths.astype(np.int32)).to(dev)
        if wl.append_one:
            kt = torch.from_numpy(inp_.k_new.view(np.int16)).to(dev).view(torch.bfloat16)
            vt = torch.from_numpy(inp_.v_new.view(np.int16)).to(dev).view(torch.bfloat16)
            si = torch.arange(B, dtype=torch.int32, device=dev)
            po = torch.from_numpy(inp_.lengths.astype(np.int32)).to(dev)
        stream = torch.cuda.current_stream(dev)
        launches_per_step = 2 if wl.append_one else 1

        def step(k, ev0=None, ev1=None, q_=None, kt_=None, vt_=None):
            c = replicas[k % len(replicas)]
            if wl.append_one:
                _lib.kvq_append(c.desc, kt if kt_ is None else kt_, vt if vt_ is None else vt_, si, po,
                                _lib.APPEND_QUANT, table, B, inp_.max_blocks, err_word=err)
            if ev0 is not None:
                ev0.record(stream)
            _lib.kvq_decode(c.desc, q if q_ is None else q_, B, Hq, dec_lens, table, inp_.max_blocks, out,
                            lse=lse, workspace=ws.buf, workspace_bytes=ws.nbytes,
                            stream_ctas=args.stream_ctas, err_word=err,
                            flags=DECODE_FLAGS)
            if ev1 is not None:
                ev1.record(stream)

        for k in range(max(args.warmup, 3)):
            step(k)
        torch.cuda.synchronize()
        # soak (untimed) so the clock sampler sees the load for >= ~1 s
        soak = 0
        if args.soak > 0:
            t_est = time.perf_counter()
            for k in range(20):
                step(k)
            torch.cuda.synchronize()
            per = max((time.perf_counter() - t_est) / 20, 1e-6)
            soak = int(min(max(args.soak / per, 0), 200000))
        K = args.steps
        # The K timed steps are captured once in a CUDA graph and replayed: the
        # host's per-call launch cost (ctypes marshalling, launch API) stays out
        # of the device timing of kernels that run for 10-400 us.  The same K
        # steps launched one by one from Python are timed beside it (eager).
        graph = None
        if not args.eager:
            try:
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    for k in range(K):
                        step(k)
                graph.replay()
                torch.cuda.synchronize()
            except Exception as e:  # reported, then timed eagerly
                graph = None
                self.graph_error = f"{type(e).__name__}: {e}"[:300]
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(self.local) as clk:
            for k in range(soak):
                step(k)
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            hold_device(torch)
            e_start.record(stream)
            if graph is not None:   # exactly K back-to-back steps, nothing else in the timed region
                graph.replay()
            else:
                for k in range(K):
                    step(k)
            e_end.record(stream)
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
        ms_total = e_start.elapsed_time(e_end)
        ms_eager = ms_total / K
        if graph is not None:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            hold_device(torch)
            e0.record(stream)
            for k in range(K):
                step(k)
            e1.record(stream)
            torch.cuda.synchronize()
            ms_eager = e0.elapsed_time(e1) / K
        # The timed steps run back to back (one decode launch each, plus the
        # append launch for append workloads).  Without an append the decode
        # kernel's average duration is the step time; with one, K decode
        # launches are timed back to back on their own.  The append alone and
        # an isolated decode launch (launch latency and tail not overlapped)
        # are reported beside it.
        n_dec = min(K, 50)
        app_ms = 0.0
        if wl.append_one:
            ea = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_dec)]
            for k in range(n_dec):
                c = replicas[k % len(replicas)]
                ea[k][0].record(stream)
                _lib.kvq_append(c.desc, kt, vt, si, po, _lib.APPEND_QUANT, table, B, inp_.max_blocks, err_word=err)
                ea[k][1].record(stream)
            torch.cuda.synchronize()
            app_ms = statistics.mean(x.elapsed_time(y) for x, y in ea)
        dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_dec)]
        for k in range(n_dec):
            step(k, *dec_ev[k])
        torch.cuda.synchronize()
        dec_iso = [a.elapsed_time(b) for a, b in dec_ev]
        if wl.append_one:
            # the decode kernel's own rate: K decode launches back to back (no append
            # in between), timed the same way as the steps
            def decodes():
                for k in range(K):
                    c = replicas[k % len(replicas)]
                    _lib.kvq_decode(c.desc, q, B, Hq, dec_lens, table, inp_.max_blocks, out, lse=lse,
                                    workspace=ws.buf, workspace_bytes=ws.nbytes, stream_ctas=args.stream_ctas,
                                    err_word=err, flags=DECODE_FLAGS)
            dgraph = None
            if graph is not None:
                dgraph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(dgraph):
                    decodes()
                dgraph.replay()
                torch.cuda.synchronize()
            ed0, ed1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            hold_device(torch)
            ed0.record(stream)
            if dgraph is not None:
                dgraph.replay()
            else:
                decodes()
            ed1.record(stream)
            torch.cuda.synchronize()
            dec_ms = ed0.elapsed_time(ed1) / K
        else:
            dec_ms = ms_total / K
        # e2e through the public API: every step copies its inputs (q, and the new
        # K/V tokens) from one pinned host staging buffer to the device in one
        # copy, runs kvq_append / kvq_decode on them, copies the output back to
        # pinned host memory and synchronizes the stream.  Each step (copy in,
        # the calls, copy out) is replayed from a CUDA graph per cache replica,
        # as a serving loop would, so the binding's per-call host cost is paid
        # once at capture; eager calls where capture is unavailable.
        nq = q.numel()
        nk = kt.numel() if wl.append_one else 0
        stage_h = torch.empty(nq + 2 * nk, dtype=torch.bfloat16).pin_memory()
        stage_h[:nq].copy_(torch.from_numpy(inp_.q.view(np.int16)).view(torch.bfloat16).reshape(-1))
        if nk:
            stage_h[nq:nq + nk].copy_(torch.from_numpy(inp_.k_new.view(np.int16)).view(torch.bfloat16).reshape(-1))
            stage_h[nq + nk:].copy_(torch.from_numpy(inp_.v_new.view(np.int16)).view(torch.bfloat16).reshape(-1))
        stage_d = torch.empty(stage_h.shape, dtype=torch.bfloat16, device=dev)
        q_dev = stage_d[:nq].view(q.shape)
        kd = stage_d[nq:nq + nk].view(kt.shape) if nk else None
        vd = stage_d[nq + nk:].view(vt.shape) if nk else None
        out_host = torch.empty((B, Hq, 128), dtype=torch.bfloat16).pin_memory()
        h2d = stage_h.numel() * 2
        d2h = out_host.numel() * 2

        def e2e_step(k):
            stage_d.copy_(stage_h, non_blocking=True)
            step(k, q_=q_dev, kt_=kd, vt_=vd)
            out_host.copy_(out, non_blocking=True)

        e2e_graphs, e2e_timing = None, "eager calls, stream synchronize per step"
        if graph is not None:
            try:
                e2e_graphs = []
                for r in range(len(replicas)):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        e2e_step(r)
                    e2e_graphs.append(g)
                for g in e2e_graphs:
                    g.replay()
                torch.cuda.synchronize()
                e2e_timing = ("cuda graph of each step (one copy in, the API calls, copy out), "
                              "stream synchronize per step")
            except Exception as e:  # capture unavailable: eager calls
                e2e_graphs = None
                e2e_timing = "eager calls (graph capture unavailable: %s)" % f"{type(e).__name__}: {e}"[:200]
        def e2e_run(k):
            if e2e_graphs:
                e2e_graphs[k % len(e2e_graphs)].replay()
            else:
                e2e_step(k)
            stream.synchronize()

        for k in range(3):  # warm-up
            e2e_run(k)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for k in range(K):
            e2e_run(k)
        e2e_s = (time.perf_counter() - t0) / K
        errbits = int(err.item())
        res = dict(ms_step=ms_total / K, ms_eager=ms_eager, timing="cuda graph of the K steps" if graph is not None
                   else "eager launches (graph capture unavailable: %s)" % getattr(self, "graph_error", "disabled"),
                   dec_ms=dec_ms, dec_ms_iso=statistics.mean(dec_iso), app_ms=app_ms,
                   e2e_s=e2e_s, e2e_timing=e2e_timing, h2d=h2d, d2h=d2h, bytes=cache_bytes_per_step(inp_),
                   replicas=len(replicas),
                   alloc=alloc, clocks=clk.summary(), launches=launches_per_step * K, err=errbits,
                   plan={"stream_ctas": plan.stream_ctas, "window_ctas": plan.window_ctas,
                         "workspace_bytes": plan.workspace_bytes})
        del replicas, ws, q, out, lse, graph, e2e_graphs, stage_d
        torch.cuda.empty_cache()
        return res

    def prefill(self, K: int):
        """kvq_prefill on the PREFILL recipe: K calls back to back, with the
        chunk's quantizing write fused into the call and without it."""
        import numpy as np
        from quantized_kv_cache_07_gb300.cache import cache_for_inputs
        from synth import Workload, make_inputs, query_rows
        torch, _lib, dev = self.torch, self.lib, self.dev
        r = PREFILL
        L = r["prefix"] + r["chunk"]
        w = Workload(r["name"], batch=r["batch"], q_heads=r["q_heads"], kv_heads=r["kv_heads"],
                     k_bits=r["k_bits"], v_bits=r["v_bits"], seq_len=L, paged=True)
        inp = make_inputs(w)
        B, Hq = w.batch, w.q_heads
        cache = cache_for_inputs(inp, dev)
        table = torch.from_numpy(inp.block_table).to(dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)

        def bits(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

        def rows(p0, p1):
            idx = np.concatenate([inp.seq_offsets[b] + np.arange(p0, p1) for b in range(B)])
            seq = np.repeat(np.arange(B, dtype=np.int32), p1 - p0)
            pos = np.tile(np.arange(p0, p1, dtype=np.int32), B)
            return idx, torch.from_numpy(seq).to(dev), torch.from_numpy(pos).to(dev)

        pi, ps, pp = rows(0, r["prefix"])
        _lib.kvq_append(cache.desc, bits(inp.k[pi]), bits(inp.v[pi]), ps, pp, _lib.APPEND_QUANT, table, B,
                        inp.max_blocks, err_word=err)
        ci, cs, cp = rows(r["prefix"], L)
        n = len(ci)
        kn, vn = bits(inp.k[ci]), bits(inp.v[ci])
        q = bits(query_rows(n, Hq, w.seed + 1))
        out = torch.empty((n, Hq, 128), dtype=torch.bfloat16, device=dev)
        split = 3 * torch.cuda.get_device_properties(dev).multi_processor_count
        nb = _lib.kvq_prefill_workspace_size(cache.desc, n, Hq, split)
        ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device=dev)
        _lib.kvq_workspace_init(ws, nb)
        times = {}
        # (fused write, path): the query-tile path with and without the write,
        # and the split-rows path (every row a query group of the decode split)
        for fused, path in ((True, _lib.PREFILL_TILES), (False, _lib.PREFILL_TILES), (False, split)):
            def call():
                _lib.kvq_prefill(cache.desc, q, Hq, cs, cp, table, B, inp.max_blocks, out,
                                 k_new=kn if fused else None, v_new=vn if fused else None, workspace=ws,
                                 workspace_bytes=nb, stream_ctas=path, err_word=err)
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            hold_device(torch)
            e0.record()
            for _ in range(K):
                call()
            e1.record()
            torch.cuda.synchronize()
            times[(fused, path)] = e0.elapsed_time(e1) / K
        per_token = token_head_bytes(w.k_bits, w.v_bits)
        req = prefill_row_bytes(r["prefix"], r["chunk"], B, w.kv_heads, per_token)
        uniq = B * w.kv_heads * per_token * L
        res = {"workload": w.name,
               "description": f"chunked prefill: {B} sequences x ({r['prefix']} cached + {r['chunk']} new "
                              f"positions), {Hq}/{w.kv_heads} heads, int{w.k_bits} K/V, paged; the new "
                              "positions are quantized into the cache and attend causally in the same call",
               "rows_per_call": n, "path": "query tiles (16 query vectors per CTA)",
               "ms_per_call": round(times[(True, _lib.PREFILL_TILES)], 6),
               "ms_per_call_attention_only": round(times[(False, _lib.PREFILL_TILES)], 6),
               "rows_per_s": round(n / (times[(True, _lib.PREFILL_TILES)] / 1e3), 1),
               "ms_per_call_split_rows_attention_only": round(times[(False, split)], 6),
               "tiles_speedup_vs_split_rows": round(times[(False, split)] / times[(False, _lib.PREFILL_TILES)], 3),
               "row_read_bytes_per_call": req,
               "cache_bytes": uniq,
               "note": "causal attention of every row over its whole prefix: the tile path reads each "
                       "(sequence, KV head) prefix once per 16 query vectors, the split-rows path once per row "
                       "(mostly from L2); neither is bound by HBM",
               "err_word": int(err.item())}
        del cache, ws, out, q, kn, vn
        torch.cuda.empty_cache()
        return res


def hold_device(torch, cycles: int = 1_000_000):
    """Queue a short device-side wait (about 0.5 ms) ahead of a timed region,
    so the host has enqueued the start event and the timed launches (a graph
    replay or K eager calls) before the device reaches them: the host's launch
    latency then stays outside the device-timed steps instead of being charged
    to the first of them."""
    torch.cuda._sleep(cycles)


def bf16_inputs(inp):
    """The same seeded bits as a plain bf16 cache (same shapes, no window, no
    factor): the same-design bf16-cache comparison."""
    import dataclasses
    wb = inp.workload.with_(k_bits=16, v_bits=16, window=0, channel_factor=False, asym=False, q_bits=16,
                            k_per_channel=False, name=inp.workload.name + "_bf16")
    return dataclasses.replace(inp, workload=wb, channel_factor=None)


def summarize(w, res, peak, peak_kind, world=1):
    """Decode-kernel roofline and step figures of one measured workload."""
    achieved = res["bytes"] / (res["dec_ms"] / 1e3) / 1e9
    kernel = "decode_asym" if w.asym else "decode"
    return {
        "workload": w.name,
        "ms_per_step": round(res["ms_step"], 6),
        "ms_per_step_eager": round(res["ms_eager"], 6),
        "timing": res["timing"],
        "steps_per_s": round(world * 1e3 / res["ms_step"], 2),
        "cache_bytes_per_step": res["bytes"],
        "effective_gbs": round(world * res["bytes"] / (res["ms_step"] / 1e3) / 1e9, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": recorded_traffic(w.name, kernel), "kernel": "kvq decode_kernel",
                     "decode_ms_back_to_back": round(res["dec_ms"], 6),
                     "append_ms_per_step": round(res["app_ms"], 6),
                     "decode_ms_isolated_launch": round(res["dec_ms_iso"], 6)},
        "e2e": {"value": round(world * res["bytes"] / res["e2e_s"] / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "ms_per_step": round(res["e2e_s"] * 1e3, 6), "timing": res["e2e_timing"]},
        "clocks": res["clocks"],
        "decode_grid": res["plan"],
        "l2": f"steps rotate over {res['replicas']} cache replicas "
              f"({res['replicas'] * res['bytes'] / 2**20:.0f} MiB >= 4x L2 or cache > L2)",
        "device_err_word": res["err"],
    }


def bf16_entry(rb, res, peak):
    g = rb["bytes"] / (rb["dec_ms"] / 1e3) / 1e9
    return {"ms_per_step": round(rb["ms_step"], 6), "decode_ms": round(rb["dec_ms"], 6),
            "decode_ms_isolated_launch": round(rb["dec_ms_iso"], 6), "bytes_per_step": rb["bytes"],
            "effective_gbs": round(g, 1), "frac_of_peak": round(g / peak, 4),
            "speedup_quant_vs_bf16": round(rb["dec_ms"] / res["dec_ms"], 4), "err_word": rb["err"]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-bf16", action="store_true", help="skip the same-design bf16-cache comparison runs")
    ap.add_argument("--no-asym", action="store_true",
                    help="skip the same-shape run in the asymmetric (scale + zero point) format")
    ap.add_argument("--asym", action="store_true",
                    help="time the workload in the asymmetric (scale + zero point) format")
    ap.add_argument("--q-bits", type=int, default=16, choices=[8, 16, 32],
                    help="query format: 8 int8 rows (integer dot), 16 fp16 (default), 32 two-part fp16")
    ap.add_argument("--no-int2", action="store_true", help="skip the 2-bit run on the int4 workload's shape")
    ap.add_argument("--no-prefill", action="store_true", help="skip the kvq_prefill measurement")
    ap.add_argument("--no-qint8", action="store_true",
                    help="skip the same-shape run with int8-quantized query rows")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only the headline workload (no per_config object)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the headline cpu_baseline (per_config entries: a third)")
    ap.add_argument("--stream-ctas", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0,
                    help="run the workload with this many sequences instead (a smaller case of the same "
                         "kernel, e.g. for a multi-pass profile); the line's workload name says so")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of a CUDA graph of the steps")
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of untimed steps before each timed region (clock sampling, steady state)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import torch
    import torch.distributed as dist

    from quantized_kv_cache_07_gb300 import _lib
    from quantized_kv_cache_07_gb300.build import build
    from synth import WORKLOADS, make_inputs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0:
        build()
    if world > 1:
        dist.barrier()
    _lib.load()

    w = WORKLOADS[args.workload]
    if args.batch > 0:
        w = w.with_(batch=args.batch, name=f"{w.name}_batch{args.batch}")
    if args.asym:
        w = w.with_(asym=True)
    if args.q_bits != 16:
        w = w.with_(q_bits=args.q_bits)
    per_config_names = [] if (args.no_per_config or world > 1) else list(ALL_WORKLOADS)
    # the oracle samples run on the host cores while the GPU is measured
    cpu_jobs = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_jobs[w.name] = start_cpu_sample(args.workload, args.cpu_budget, asym=w.asym, qbits=w.q_bits,
                                            batch=args.batch)
        for n in per_config_names:
            if n != args.workload or w.asym or w.q_bits != 16:
                cpu_jobs[n + "/per_config"] = start_cpu_sample(n, args.cpu_budget / 3)

    dev = torch.device("cuda", local)
    arm = GpuArm(args, dev, world, local)
    peak, peak_kind = measured_peaks()

    def allmax(x):
        return max_over_ranks(x, world, dev)

    inp = make_inputs(w)
    res = arm.run(inp)
    ms_step = allmax(res["ms_step"])
    e2e_s = allmax(res["e2e_s"])
    bytes_step = res["bytes"]
    value = world * bytes_step / (ms_step / 1e3) / 1e9
    achieved = bytes_step / (res["dec_ms"] / 1e3) / 1e9

    bf16 = None
    if not args.no_bf16 and w.k_bits != 16:
        bf16 = dict(workload=w.name + "_bf16", **bf16_entry(arm.run(bf16_inputs(inp)), res, peak))

    asym = None
    if not args.no_asym and w.k_bits != 16 and not w.asym:
        import dataclasses
        wa = w.with_(asym=True, name=w.name + "_asym")
        ra = arm.run(dataclasses.replace(inp, workload=wa))     # same bits, scale + zero point
        asym = {"workload": wa.name, "ms_per_step": ra["ms_step"], "decode_ms": ra["dec_ms"],
                "decode_ms_isolated_launch": ra["dec_ms_iso"], "bytes_per_step": ra["bytes"],
                "effective_gbs": ra["bytes"] / (ra["dec_ms"] / 1e3) / 1e9,
                "frac_of_peak": ra["bytes"] / (ra["dec_ms"] / 1e3) / 1e9 / peak,
                "time_vs_symmetric": ra["dec_ms"] / res["dec_ms"], "err_word": ra["err"]}

    qint8 = None
    if not args.no_qint8 and w.k_bits != 16 and w.q_bits != 8 and not (w.channel_factor and w.window):
        import dataclasses
        wq = w.with_(q_bits=8, name=w.name + "_qint8")
        rq = arm.run(dataclasses.replace(inp, workload=wq))     # same bits, int8 query rows
        qint8 = {"workload": wq.name, "ms_per_step": rq["ms_step"], "decode_ms": rq["dec_ms"],
                 "bytes_per_step": rq["bytes"], "effective_gbs": rq["bytes"] / (rq["dec_ms"] / 1e3) / 1e9,
                 "frac_of_peak": rq["bytes"] / (rq["dec_ms"] / 1e3) / 1e9 / peak,
                 "time_vs_bf16_query": rq["dec_ms"] / res["dec_ms"], "err_word": rq["err"]}

    # every named workload, one after another (rank 0 at one GPU)
    per_config = {}
    for n in per_config_names:
        if n == args.workload and not w.asym and w.q_bits == 16:
            entry = summarize(w, res, peak, peak_kind)
            entry["bf16_same_design"] = bf16
        else:
            wn = WORKLOADS[n]
            inn = make_inputs(wn)
            rn = arm.run(inn)
            entry = summarize(wn, rn, peak, peak_kind)
            entry["bf16_same_design"] = (None if args.no_bf16 else
                                         dict(workload=n + "_bf16", **bf16_entry(arm.run(bf16_inputs(inn)), rn,
                                                                                 peak)))
            if n == INT2_SHAPE and not args.no_int2:
                import dataclasses
                w2 = wn.with_(k_bits=2, v_bits=2, name=n.replace("int4", "int2"))
                r2 = arm.run(dataclasses.replace(inn, workload=w2))     # same bits, 2-bit token groups
                entry["int2_same_shape"] = {
                    "workload": w2.name, "ms_per_step": round(r2["ms_step"], 6), "bytes_per_step": r2["bytes"],
                    "effective_gbs": round(r2["bytes"] / (r2["dec_ms"] / 1e3) / 1e9, 1),
                    "frac_of_peak": round(r2["bytes"] / (r2["dec_ms"] / 1e3) / 1e9 / peak, 4),
                    "time_vs_int4": round(r2["dec_ms"] / rn["dec_ms"], 4), "err_word": r2["err"]}
            del inn
        per_config[n] = entry
    prefill = None if (args.no_prefill or world > 1) else arm.prefill(args.steps)

    line = {
        "metric": "quantized-KV decode attention: effective HBM GB/s (% of peak), steps/s",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms_step, 6),
        "steps_per_s": round(world * 1e3 / ms_step, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "s8/s4 codes, f16 mma, f32 accumulate" if w.k_bits != 16 else "bf16 mma, f32 accumulate",
        "data": "synthetic (seeded), cache resident in HBM",
        "config": {"workload": w.name, "description": w.description, "batch": w.batch, "q_heads": w.q_heads,
                   "kv_heads": w.kv_heads, "head_dim": w.head_dim, "k_bits": w.k_bits, "v_bits": w.v_bits,
                   "window": w.window, "paged": w.paged, "append_one": w.append_one,
                   "format": "asymmetric (scale + zero point)" if w.asym else "symmetric (scale)",
                   "query": {8: "int8 rows, integer dot", 16: "fp16", 32: "two-part fp16 (hi + lo)"}[w.q_bits],
                   "cache_bytes_per_step": bytes_step, "allocated_cache_bytes": res["alloc"],
                   "l2": f"steps rotate over {res['replicas']} cache replicas "
                         f"({res['replicas'] * bytes_step / 2**20:.0f} MiB >= 4x L2 or cache > L2)",
                   "parallelism": f"replicas x{world}", "decode_grid": res["plan"], "timing": res["timing"],
                   "decode_flags": "KVQ_DECODE_GEOMETRY_READY" if DECODE_FLAGS else "0",
                   "ms_per_step_eager": round(res["ms_eager"], 6)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": recorded_traffic(w.name, "decode_asym" if w.asym else "decode"),
                     "kernel": "kvq decode_kernel",
                     "decode_ms_back_to_back": round(res["dec_ms"], 6),
                     "append_ms_per_step": round(res["app_ms"], 6),
                     "decode_ms_isolated_launch": round(res["dec_ms_iso"], 6)},
        "e2e": {"value": round(world * bytes_step / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "ms_per_step": round(e2e_s * 1e3, 6), "timing": res["e2e_timing"]},
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "bf16_same_design": bf16,
        "asym_same_shape": asym,
        "qint8_same_shape": qint8,
        "prefill": prefill,
        "device_err_word": res["err"],
    }
    if per_config:
        line["per_config"] = per_config
    for key, proc in cpu_jobs.items():
        name = key.split("/")[0]
        try:
            entry = cpu_baseline_entry(finish_cpu_sample(proc), name)
        except Exception as e:  # reported, not fatal
            entry = {"value": None, "unit": "GB/s", "cores": 1, "host_cores": host_cores(), "kind": "oracle",
                     "sample": f"failed: {e}"}
        if key.endswith("/per_config"):
            per_config[name]["cpu_baseline"] = entry
        else:
            line["cpu_baseline"] = entry
            if name in per_config:
                per_config[name]["cpu_baseline"] = entry
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def reference_arm(args, rank, world):
    """The float64 CPU oracle as the reference arm: rank 0 only."""
    if rank != 0:
        return
    from synth import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.batch > 0:
        w = w.with_(batch=args.batch, name=f"{w.name}_batch{args.batch}")
    K = args.steps
    # bounded: about 60 s of oracle work for the whole timed run, split over K steps
    per_step_budget = min(60.0 / max(K, 1), 5.0)
    d = run_cpu_sample(args.workload, per_step_budget * K, batch=args.batch)
    gbs = d["bytes"] / d["seconds"] / 1e9
    ms = d["seconds"] / K * 1e3
    line = {
        "impl": "reference",
        "metric": "quantized-KV decode attention: effective HBM GB/s (% of peak), steps/s",
        "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": w.name, "description": w.description,
                   "sample": "each step: a bounded sample of (sequence, kv_head) units"},
        "cpu_baseline": cpu_baseline_entry(d, w.name),
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
