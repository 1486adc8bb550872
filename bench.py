"""Benchmark: decode-attention tokens/s and achieved HBM GB/s on one GB300.

A step is one pass of the whole hot path over one batch: the new K/V row of
every (sequence, kv head) is appended and the decode runs over the grown cache,
in one fused launch (``decode_attn_append``; ``--separate-append`` times
``kv_append`` followed by ``decode_attn`` instead).  The
step cycles through 16 consecutive positions (context n+1 ... n+16, as in
the MHA fp32 workload's 16 append+decode steps), so the context length is the
same however many steps run.  Inputs are seeded synthetic tensors resident in
HBM before timing; K/V copies are rotated so that the cache bytes touched
between two reads of the same copy exceed 4x the L2 size.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead.  Under torchrun every rank runs an independent
replica (its own batch; no collective on the data path); timing is the max
over ranks and ``value`` counts all ranks' tokens.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from decode_attention_kv_split_gb300 import accounting, workloads as W  # noqa: E402

METRIC = "decode-attn tokens/s and achieved HBM GB/s (% of GB300 peak) vs context"
L2_BYTES = 129 * 1024 * 1024
CYCLE = 16
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_family(w) -> str:
    """Source file of the split kernel a workload runs."""
    if W.is_q8(w):
        return "decode_q8.cu"
    if w.dtype == torch.float32:
        return "decode_fp32.cu"
    if w.d_k == 128 and w.d_v == 128 and w.h_q // w.h_kv > 8:
        return "decode_tc5.cu"
    return "decode_bf16.cu"


def kernel_source_hash(w) -> str:
    """Hash of the sources that decide a workload's decode launches: the split
    kernel's file, the shared device code, the combine and the host planner."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_kv_split_gb300", "csrc")
    for fn in ("common.cuh", "combine.cu", "api.cu", kernel_family(w)):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(w):
    """DRAM bytes per decode launch from a committed ncu capture, if it was taken
    on the current kernel sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(w.name)
        if e and e.get("kernel_source_hash") == kernel_source_hash(w):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.reader.join(timeout=2)
        return self.summary(self.t0, self.t1)

    def summary(self, t0, t1):
        """Median SM clock and the throttle reasons seen between host times t0 and t1."""
        if self.proc is None:
            return None
        rows = []
        for ts, line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        if not rows:
            return None
        inwin = [r for r in rows if t0 is not None and t0 <= r[0] <= (t1 or 1e30)]
        use = inwin if inwin else rows
        sm = sorted(r[1] for r in use)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if "Active" in v
                          and "Not" not in v})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inwin)}


def dist_setup(backend: str | None = None):
    """Join the torchrun job (one replica per GPU).  Returns (world, rank, local)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_rate(local_ms: float, world: int, units_per_rank: int, steps: int):
    """Whole-job rate of `world` independent replicas: every rank processed
    `units_per_rank` units in each of `steps` steps, and the job took as long as
    its slowest rank.  Returns (ms per step, units/s over all ranks)."""
    total_ms = max_over_ranks(local_ms, world)
    ms_per_step = total_ms / steps
    return ms_per_step, world * units_per_rank / (ms_per_step / 1e3)


def padded(w):
    """The workload as the bench allocates it: room for the CYCLE appended rows."""
    return W.custom(name=w.name, B=w.B, h_q=w.h_q, h_kv=w.h_kv, d_k=w.d_k, d_v=w.d_v, n=w.n,
                    n_max=w.n_max + CYCLE, dtype=w.dtype, kv_std=w.kv_std, ragged=w.ragged,
                    num_splits=w.num_splits, description=w.description)


def decode_bytes_of(w, lens) -> int:
    """Algorithmic bytes of one decode over the given lengths."""
    if W.is_q8(w):
        return accounting.decode_bytes_q8(lens, w.h_q, w.h_kv, w.d_k, w.d_v)
    es = 2 if w.dtype == torch.bfloat16 else 4
    return accounting.decode_bytes(lens, w.h_q, w.h_kv, w.d_k, w.d_v, es)


def rotation(w):
    """(K/V copies the bench rotates through, bytes one step touches): enough copies
    that the cache bytes read between two uses of one copy exceed 4x the L2."""
    kv_touch = decode_bytes_of(w, (W.seq_lens(w) + CYCLE).tolist())
    return int(min(64, max(1, math.ceil(4 * L2_BYTES / kv_touch)))), kv_touch


def workload_config(wb):
    """The ``config`` object of a bench line: depends on the workload alone, so that
    both arms print the same one."""
    n_rot, kv_bytes = rotation(wb)
    cfg = {"workload": wb.description, "name": wb.name, "B": wb.B, "h_q": wb.h_q,
           "h_kv": wb.h_kv, "d_k": wb.d_k, "d_v": wb.d_v, "n_start": wb.n,
           "context": f"n+1 .. n+{CYCLE}", "n_max_allocated": wb.n_max,
           "kv_dtype": str(wb.dtype).replace("torch.", ""),
           "num_splits": {0: "auto", -1: "balanced"}.get(wb.num_splits, wb.num_splits),
           "parallelism": "replicas (one per GPU)",
           "tokens_per_step": wb.B}
    if wb.ragged:
        cfg["lengths"] = f"uniform in [{wb.ragged[0]}, {wb.ragged[1]}] (seed 3)"
    if n_rot * kv_bytes >= 4 * L2_BYTES and n_rot == 1:
        cfg["l2"] = (f"inputs larger than L2: one K/V cache of {kv_bytes / 1e6:.0f} MB per step "
                     f"(>= 4x the {L2_BYTES >> 20} MiB L2)")
    elif n_rot * kv_bytes >= 4 * L2_BYTES:
        cfg["l2"] = (f"inputs larger than L2: {n_rot} rotating K/V copies of "
                     f"{kv_bytes / 1e6:.0f} MB each (>= 4x the {L2_BYTES >> 20} MiB L2 "
                     "between reuses)")
    else:
        cfg["l2"] = (f"L2-resident: {n_rot} K/V copies of {kv_bytes / 1e6:.2f} MB; "
                     "latency only, GB/s not meaningful")
    return cfg


# --------------------------------------------------------------------------- oracle timing
class OracleStep:
    """The CPU oracle run on the bench's own workload: one step appends the new K/V
    row of every (sequence, kv head) and decodes every query head over the grown
    cache, exactly the step the GPU arm times (oracle ``kv_append`` then
    ``decode``, fp64 arithmetic on the same rounded inputs).  An 8-bit cache is
    timed on its float32 values before quantization: the oracle's decode does
    the same work on any values."""

    def __init__(self, w):
        import numpy as np
        import oracle

        self.o = oracle.get()
        self.wb = wb = padded(w)
        self.lens0 = W.seq_lens(wb).numpy().astype(np.int32)
        vals = torch.float32 if W.is_q8(wb) else wb.dtype
        K, V = W.cache(dataclasses.replace(wb, dtype=vals))
        self.K = np.ascontiguousarray(K.float().numpy())
        self.V = np.ascontiguousarray(V.float().numpy())
        del K, V
        self.q = np.ascontiguousarray(W.query(wb).float().numpy())
        rows = [W.new_rows(wb, t) for t in range(CYCLE)]
        self.rows = [(np.ascontiguousarray(k.float().numpy()),
                      np.ascontiguousarray(v.float().numpy())) for k, v in rows]
        self.cores = self.o.max_threads()

    def step(self, i: int, threads: int, seqs=None):
        """Append at position n + (i mod CYCLE), decode over one row more.  ``seqs``
        limits the step to the first ``seqs`` sequences (a bounded sample)."""
        c = i % CYCLE
        kn, vn = self.rows[c]
        pos = self.lens0 + c
        self.o.kv_append(kn, vn, self.K, self.V, pos)
        b = self.wb.B if seqs is None else seqs
        self.o.decode(self.q[:b], self.K[:b], self.V[:b], (pos + 1)[:b], self.wb.scale,
                      threads=threads)

    def rows_of(self, seqs=None) -> float:
        b = self.wb.B if seqs is None else seqs
        return float(self.lens0[:b].sum()) + b * (CYCLE + 1) / 2


def oracle_baseline(w, seconds: float):
    """cpu_baseline of a bench line: the oracle timed on the host cores on the
    workload itself (whole steps, all cores), plus a one-core figure from a
    one-sequence sample of a step, scaled to the whole step by its rows."""
    st = OracleStep(w)
    cores = st.cores
    st.step(0, cores)  # first touch of the arrays
    t0 = time.perf_counter()
    steps = 0
    while steps < 1 or time.perf_counter() - t0 < seconds / 2:
        st.step(1 + steps, cores)
        steps += 1
    el = time.perf_counter() - t0
    tok_s = st.wb.B * steps / el
    t1 = time.perf_counter()
    st.step(0, 1, seqs=1)
    el1 = time.perf_counter() - t1
    tok_s_1 = st.wb.B / (el1 * st.rows_of() / st.rows_of(1))
    sample = (f"oracle kv_append + decode (fp64) on the workload itself: {steps} whole step(s) "
              f"on {cores} threads in {el:.2f} s; one-core figure from sequence 0 of a step "
              f"({el1:.2f} s) scaled to the step's rows")
    return {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": sample, "value_1core": tok_s_1}


def run_reference(args, w, world, rank):
    """The reference arm: the CPU oracle, as it stands, on the host cores (rank 0
    only), over the same workload, metric and config as the GPU arm."""
    if rank != 0:
        return
    st = OracleStep(w)
    cores = st.cores
    for i in range(args.warmup):
        st.step(i, cores)
    t0 = time.perf_counter()
    for i in range(args.steps):
        st.step(args.warmup + i, cores)
    el = time.perf_counter() - t0
    value = st.wb.B * args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(st.wb),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"oracle kv_append + decode (fp64), {args.steps} whole "
                                       f"steps of the workload on {cores} threads"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# --------------------------------------------------------------------------- our arm
class Harness:
    """Device-resident inputs of one workload and the step that the bench times."""

    def __init__(self, w, rank: int, fused: bool, gpu_cache: bool = False):
        from decode_attention_kv_split_gb300 import api

        self.api = api
        dev = torch.device("cuda", torch.cuda.current_device())
        torch.manual_seed(rank)
        wb = padded(w)
        n_max = wb.n_max
        seed = 1000 * rank
        lens0 = W.seq_lens(wb, seed)
        self.q8 = W.is_q8(w)
        es = 1 if self.q8 else (2 if w.dtype == torch.bfloat16 else 4)
        row_bytes = (w.d_k + 4) if self.q8 else w.d_k * es  # an 8-bit row carries its scale
        self.w, self.es = w, es
        n_rot, kv_touch = rotation(wb)
        cache_bytes = 2 * wb.B * wb.h_kv * n_max * row_bytes
        free = torch.cuda.mem_get_info(dev)[0]
        n_rot = int(max(1, min(n_rot, (0.6 * free) // cache_bytes)))

        K0, V0 = W.cache(wb, seed, device=dev if gpu_cache else "cpu")
        K0, V0 = K0.to(dev), V0.to(dev)
        if self.q8:  # 8-bit cache: codes + row scales, quantized by the library's kernel
            (K0, ks0), (V0, vs0) = api.kv_quantize(K0, w.dtype), api.kv_quantize(V0, w.dtype)
            first = (K0, V0, ks0, vs0)
        else:
            first = (K0, V0)
        self.caches = [first] + [tuple(t.clone() for t in first) for _ in range(n_rot - 1)]
        del K0, V0, first
        self.q = W.query(wb, seed).to(dev)
        rows = [W.new_rows(wb, t, seed) for t in range(CYCLE)]
        if self.q8:
            kq = [api.kv_quantize(k.to(dev), w.dtype) for k, _ in rows]
            vq = [api.kv_quantize(v.to(dev), w.dtype) for _, v in rows]
            self.k_new, self.k_new_scale = [c for c, _ in kq], [s for _, s in kq]
            self.v_new, self.v_new_scale = [c for c, _ in vq], [s for _, s in vq]
        else:
            self.k_new = [k.to(dev) for k, _ in rows]
            self.v_new = [v.to(dev) for _, v in rows]
        self.pos_t = [(lens0 + t).to(torch.int32).to(dev) for t in range(CYCLE)]
        self.lens_t = [(lens0 + t + 1).to(torch.int32).to(dev) for t in range(CYCLE)]
        self.out = torch.empty((wb.B, wb.h_q, wb.d_v), dtype=torch.float32, device=dev)
        self.splits = api.resolve_splits(wb.B, wb.h_q, wb.h_kv, wb.d_k, wb.d_v, n_max, wb.dtype,
                                         w.num_splits)
        ws_bytes = api.workspace_bytes(wb.B, wb.h_q, wb.h_kv, wb.d_k, wb.d_v, n_max, wb.dtype,
                                       w.num_splits)
        self.ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        self.wb, self.lens0 = wb, lens0
        self.n_rot, self.kv_touch, self.fused = n_rot, kv_touch, fused

    def _decode_bytes(self, lens) -> int:
        w = self.w
        if self.q8:
            return accounting.decode_bytes_q8(lens, w.h_q, w.h_kv, w.d_k, w.d_v)
        return accounting.decode_bytes(lens, w.h_q, w.h_kv, w.d_k, w.d_v, self.es)

    def step(self, i, qq=None, kn=None, vn=None, kns=None, vns=None):
        """One pass of the hot path: append row pos of every kv head, decode over pos+1."""
        api, w = self.api, self.w
        c = i % CYCLE
        qq = self.q if qq is None else qq
        kn = self.k_new[c] if kn is None else kn
        vn = self.v_new[c] if vn is None else vn
        if self.q8:
            K, V, ks, vs = self.caches[i % self.n_rot]
            kns = self.k_new_scale[c] if kns is None else kns
            vns = self.v_new_scale[c] if vns is None else vns
            if self.fused:
                api.decode_attn_q8_append(qq, kn, vn, kns, vns, K, V, ks, vs, self.pos_t[c],
                                          out=self.out, num_splits=w.num_splits, workspace=self.ws)
            else:
                api.kv_append_q8(kn, vn, kns, vns, K, V, ks, vs, self.pos_t[c])
                api.decode_attn_q8(qq, K, V, ks, vs, self.lens_t[c], out=self.out,
                                   num_splits=w.num_splits, workspace=self.ws)
            return
        K, V = self.caches[i % self.n_rot]
        if self.fused:
            api.decode_attn_append(qq, kn, vn, K, V, self.pos_t[c], out=self.out,
                                   num_splits=w.num_splits, workspace=self.ws)
        else:
            api.kv_append(kn, vn, K, V, self.pos_t[c])
            api.decode_attn(qq, K, V, self.lens_t[c], out=self.out, num_splits=w.num_splits,
                            workspace=self.ws)

    def step_bytes(self) -> int:
        """Algorithmic HBM bytes of one step at the mean context of the 16-step cycle."""
        w = self.w
        mean_lens = [int(n) + (CYCLE + 1) / 2 for n in self.lens0.tolist()]
        dec = self._decode_bytes(mean_lens)
        app = (accounting.append_bytes_q8(w.B, w.h_kv, w.d_k, w.d_v) if self.q8
               else accounting.append_bytes(w.B, w.h_kv, w.d_k, w.d_v, self.es))
        # the fused call reads the new row once (from k_new/v_new) and writes it once
        return dec + app // 2 if self.fused else dec + app

    def capture(self, K: int):
        """Record K consecutive steps into one CUDA graph (the way a serving loop
        removes the host launch cost).  Returns (graph, kernels per replay)."""
        api = self.api
        g = torch.cuda.CUDAGraph()
        n0 = api.launch_count()
        with torch.cuda.graph(g):
            for i in range(K):
                self.step(i)
        torch.cuda.synchronize()
        return g, api.launch_count() - n0

    def time_steps(self, K: int, world: int = 1, graph=None) -> float:
        """Device time in ms of K consecutive steps, from one CUDA event pair on the
        stream, bracketed by a barrier and a device synchronize on both sides: a
        replay of `graph` (K steps recorded by capture()), or K eager calls."""
        ev_start = torch.cuda.Event(enable_timing=True)
        ev_end = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        # Keep the GPU busy (outside the timed region) while the host queues the
        # steps, so that host launch latency does not leak into the timing.
        torch.cuda._sleep(int(2e6 if graph is not None else 2e6 + 8e4 * K))
        ev_start.record(self.stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(K):
                self.step(i)
        ev_end.record(self.stream)
        torch.cuda.synchronize()
        barrier(world)
        return ev_start.elapsed_time(ev_end)

    def time_windows(self, K: int, world: int, graph=None, min_s: float = 0.8):
        """Repeated K-step windows (each timed as time_steps does) until about
        `min_s` seconds of device time have passed, at least 5 and at most 400
        windows, the same count on every rank.  Returns the window times in ms."""
        first = self.time_steps(K, world, graph)
        reps = int(min(400, max(5, math.ceil(min_s * 1e3 / max(first, 1e-3)))))
        reps = int(max_over_ranks(reps, world))
        return [self.time_steps(K, world, graph) for _ in range(reps)]


def run_ours(args, w, world, rank, local):
    from decode_attention_kv_split_gb300 import api

    h = Harness(w, rank, fused=not args.separate_append)
    step, stream, fused, splits = h.step, h.stream, h.fused, h.splits
    q, k_new, v_new, out = h.q, h.k_new, h.v_new, h.out
    wb, n_rot, kv_touch = h.wb, h.n_rot, h.kv_touch
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    K = args.steps
    graph = None
    if not args.eager:
        graph, launches_per_window = h.capture(K)
        h.time_steps(K, world, graph)  # first replay: uploads the graph
    launches0 = api.launch_count()
    if sampler:
        sampler.mark(True)
    windows = h.time_windows(K, world, graph)
    if sampler:
        sampler.mark(False)
    if args.eager:
        launches = api.launch_count() - launches0
        launches_per_window = launches // (len(windows) + 1)
    else:
        launches = launches_per_window * len(windows)
    del graph
    local_ms = sorted(windows)[len(windows) // 2]  # median window
    ms_per_step, tokens_per_s = replica_rate(local_ms, world, w.B, K)
    clocks = sampler.stop() if sampler else None

    # ---- end to end: pinned host inputs in, result out, every step
    # Per step: q and the new rows (with their scales for an 8-bit cache), packed
    # into one pinned host buffer per cycle position and copied in with one H2D
    # copy; the result is read back into pinned host memory and the host waits
    # for it before the next step (a decode loop needs each token's result).
    rows_d = [k_new, v_new] + ([h.k_new_scale, h.v_new_scale] if h.q8 else [])
    parts = [q] + [ts[0] for ts in rows_d]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    stage_d = torch.empty(total, dtype=torch.uint8, device=q.device)

    def view(buf, t, off):
        return buf[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    dev_views = [view(stage_d, t, o) for t, o in zip(parts, offs)]
    stage_h = []
    for c in range(CYCLE):
        hb = torch.empty(total, dtype=torch.uint8).pin_memory()
        for t, o, src in zip(parts, offs, [q] + [ts[c] for ts in rows_d]):
            view(hb, t, o).copy_(src.cpu())
        stage_h.append(hb)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    q_d, bufs = dev_views[0], dev_views[1:]

    def e2e_body(i):
        stage_d.copy_(stage_h[i % CYCLE], non_blocking=True)
        step(i, q_d, *bufs)
        out_h.copy_(out, non_blocking=True)

    e2e_steps = min(2000, max(K, 200))
    # (a) each step a replay of a CUDA graph holding its H2D copy, its C-ABI
    # call and its D2H copy (how a serving loop issues decode steps), then a
    # host wait for the result
    period = CYCLE * h.n_rot // math.gcd(CYCLE, h.n_rot)
    e2e_graphs = []
    for i in range(period):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e2e_body(i)
        e2e_graphs.append(g)
    torch.cuda.synchronize()

    def run_e2e(use_graph: bool) -> float:
        for i in range(min(args.warmup, 8)):
            if use_graph:
                e2e_graphs[i % period].replay()
            else:
                e2e_body(i)
            stream.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            if use_graph:
                e2e_graphs[i % period].replay()
            else:
                e2e_body(i)
            stream.synchronize()
        return replica_rate(1e3 * (time.perf_counter() - t0), world, w.B, e2e_steps)[1]

    e2e_rate = run_e2e(True)
    e2e_eager = run_e2e(False)  # (b) the same, one eager C-ABI call per step
    del e2e_graphs
    h2d = sum(t.numel() * t.element_size() for t in parts)
    d2h = out.numel() * out.element_size()

    if rank != 0:
        return
    # ---- accounting
    step_bytes = h.step_bytes()
    peak, peak_kind = peaks()
    achieved = step_bytes / (ms_per_step / 1e3) / 1e9
    traffic = recorded_traffic(w)
    bytes_str = f"{step_bytes / 1e6:.1f} MB per step"
    if h.n_rot * h.kv_touch < 4 * L2_BYTES:
        bytes_str += " (L2-resident)"

    cpu = oracle_baseline(w, args.cpu_seconds) if args.cpu_seconds > 0 else None
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("f16 (8-bit codes, fp32 scales)" if h.q8
                  else "f32" if w.dtype == torch.float32 else "bf16"),
        "data": "synthetic", "config": workload_config(wb),
        "hbm_gbs": achieved,
        "hbm_frac_of_8tbs": achieved / 8000.0,
        "step": "decode_attn_append (fused append + decode)" if fused
        else "kv_append then decode_attn",
        "max_splits": splits,
        "roofline": {"bound": "hbm",
                     "kernel": ("split_decode kernel with fused append" if fused
                                else "kv_append + split_decode kernels")
                     + (" (+ PDL LSE combine)" if splits > 1 else ""),
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} copy bandwidth",
                     "timing": "CUDA events on the launching stream around each window of K "
                               "steps; median window",
                     "traffic": traffic, "algorithmic_bytes": step_bytes, "per": bytes_str},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_rate, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "sync": "host waits for each step's result",
                "launch": "per step: a CUDA-graph replay of the H2D copy from pinned host memory, "
                          "the C-ABI call and the D2H copy of out",
                "value_eager": e2e_eager},
        "gpu_launches": launches,
        "gpu_launches_per_step": launches_per_window / K,
        "launch": ("eager: one C-ABI call per step" if args.eager else
                   "the K steps recorded once through the C-ABI into a CUDA graph, "
                   "replayed once per timed window"),
        "windows": {"count": len(windows), "steps_each": K,
                    "ms_min": min(windows), "ms_median": local_ms, "ms_max": max(windows),
                    "value_from": "median window"},
        "clocks": clocks,
    }
    print(json.dumps(line))


SWEEP_CONTEXTS = (1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072)
SWEEP_SHAPES = ("gqa_llama3_8b", "mqa_g32", "long_llama2_70b", "mha_fp32", "long_llama2_70b_fp8")


def run_sweep(args):
    """Tokens/s and HBM GB/s against context length: every listed workload shape at
    every context in ``--contexts``, all sequences at the same length, the fused step,
    splits as ``--splits`` says (default: the library's choice).  One JSON line per
    point; the K/V caches are drawn by a CUDA generator (timing only, no parity)."""
    import dataclasses

    peak, peak_kind = peaks()
    contexts = [int(c) for c in args.contexts.split(",")]
    shapes = args.sweep.split(",") if args.sweep != "all" else list(SWEEP_SHAPES)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    for name in shapes:
        for n in contexts:
            w = dataclasses.replace(W.WORKLOADS[name], n=n, n_max=n, ragged=None,
                                    num_splits=args.splits or 0)
            h = Harness(w, 0, fused=True, gpu_cache=True)
            for i in range(args.warmup):
                h.step(i)
            probe_ms = h.time_steps(20) / 20
            K = int(min(args.steps, max(50, 300.0 / probe_ms)))
            graph = None
            if not args.eager:
                graph, _ = h.capture(K)
                h.time_steps(K, 1, graph)
            t0 = time.time()
            ms = h.time_steps(K, 1, graph) / K
            del graph
            clocks = sampler.summary(t0, time.time())
            gbs = h.step_bytes() / (ms / 1e3) / 1e9
            print(json.dumps({
                "sweep": name, "context": f"{n + 1}..{n + CYCLE}", "n": n, "B": w.B,
                "h_q": w.h_q, "h_kv": w.h_kv, "d": w.d_k,
                "kv_dtype": str(w.dtype).replace("torch.", ""), "steps": K,
                "us_per_step": 1e3 * ms, "tokens_per_s": w.B / (ms / 1e3), "hbm_gbs": gbs,
                "frac": gbs / peak, "peak": peak, "peak_kind": peak_kind,
                "max_splits": h.splits, "n_rot": h.n_rot, "clocks": clocks,
                "launch": "eager" if args.eager else "cuda graph"}), flush=True)
            del h
            torch.cuda.empty_cache()
    sampler.stop()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_llama2_70b", choices=sorted(W.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--separate-append", action="store_true",
                    help="run kv_append and decode_attn as two launches instead of the fused call")
    ap.add_argument("--splits", type=int, default=None,
                    help="override the workload's splits per sequence (0 = library's choice)")
    ap.add_argument("--eager", action="store_true",
                    help="time K eager C-ABI calls instead of one CUDA-graph replay of them")
    ap.add_argument("--sweep", default=None,
                    help="context sweep instead of the bench line: 'all' or a comma list of "
                         "workload shapes")
    ap.add_argument("--contexts", default=",".join(str(c) for c in SWEEP_CONTEXTS),
                    help="contexts of the sweep (comma list)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = W.WORKLOADS[args.workload]
    if args.splits is not None:
        import dataclasses
        w = dataclasses.replace(w, num_splits=args.splits)
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, w, int(os.environ.get("WORLD_SIZE", "1")), rank)
        return
    world, rank, local = dist_setup()
    if args.sweep:
        if rank == 0:
            run_sweep(args)
    else:
        run_ours(args, w, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
