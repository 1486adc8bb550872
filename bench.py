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


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_kv_split_gb300", "csrc")
    for fn in ("common.cuh", "decode_bf16.cu", "decode_fp32.cu", "decode_tc5.cu"):  # split kernels
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per decode launch from a committed ncu capture, if it was taken
    on the current kernel sources; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("kernel_source_hash") == kernel_source_hash():
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


def workload_config(w, n_rot: int, kv_bytes: int):
    cfg = {"workload": w.description, "name": w.name, "B": w.B, "h_q": w.h_q, "h_kv": w.h_kv,
           "d_k": w.d_k, "d_v": w.d_v, "n_start": w.n, "context": f"n+1 .. n+{CYCLE}",
           "n_max_allocated": w.n_max + CYCLE, "kv_dtype": str(w.dtype).replace("torch.", ""),
           "num_splits": {0: "auto", -1: "balanced"}.get(w.num_splits, w.num_splits),
           "parallelism": "replicas (one per GPU)",
           "tokens_per_step": w.B}
    if w.ragged:
        cfg["lengths"] = f"uniform in [{w.ragged[0]}, {w.ragged[1]}] (seed 3)"
    if n_rot * kv_bytes >= 4 * L2_BYTES:
        cfg["l2"] = (f"{n_rot} rotating K/V copies of {kv_bytes / 1e6:.0f} MB each "
                     f"(>= 4x the {L2_BYTES >> 20} MiB L2 between reuses)")
    else:
        cfg["l2"] = (f"L2-resident: {n_rot} K/V copies of {kv_bytes / 1e6:.2f} MB; "
                     "latency only, GB/s not meaningful")
    return cfg


# --------------------------------------------------------------------------- oracle timing
def oracle_step_sample(w, budget_s: float, threads: int):
    """Time the oracle's decode on a bounded sample of the workload's (b, h)
    heads at context n+1.  Returns (tokens/s equivalent, sample text, cores)."""
    import numpy as np
    import oracle

    o = oracle.get()
    cores = min(threads, o.max_threads())
    lens = W.seq_lens(w)
    q = W.query(w).float().numpy()
    # one kv head's rows are shared by its group; sample whole groups of heads
    n1 = int(lens[0]) + 1
    g = np.random.default_rng(0)
    Kh = g.standard_normal((n1, w.d_k)).astype(np.float32)
    Vh = g.standard_normal((n1, w.d_v)).astype(np.float32)
    t0 = time.perf_counter()
    heads = 0
    while True:
        o.decode_head(q[0, heads % w.h_q], Kh, Vh, w.scale)
        heads += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    # every token needs B*h_q heads at this context length (ragged: mean length)
    mean_len = float(lens.double().mean()) + 1
    heads_per_token = w.h_q * (mean_len / n1)
    tok_s = heads / heads_per_token / el
    return tok_s, (f"oracle decode_head (fp64, 1 thread) on {heads} single heads at n={n1} "
                   f"for {el:.1f} s, scaled to B*h_q heads per token at mean context "
                   f"{mean_len:.0f}"), 1


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    budget = max(0.02, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_step_sample(w, budget / 4, 1)
    t0 = time.perf_counter()
    vals = []
    sample = ""
    for _ in range(args.steps):
        v, sample, cores = oracle_step_sample(w, budget, 1)
        vals.append(v)
    el = time.perf_counter() - t0
    value = sum(vals) / len(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, 1, 0),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
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
        n_max = w.n_max + CYCLE
        wb = W.custom(name=w.name, B=w.B, h_q=w.h_q, h_kv=w.h_kv, d_k=w.d_k, d_v=w.d_v, n=w.n,
                      n_max=n_max, dtype=w.dtype, kv_std=w.kv_std, ragged=w.ragged,
                      num_splits=w.num_splits, description=w.description)
        seed = 1000 * rank
        lens0 = W.seq_lens(wb, seed)
        self.q8 = W.is_q8(w)
        es = 1 if self.q8 else (2 if w.dtype == torch.bfloat16 else 4)
        row_bytes = (w.d_k + 4) if self.q8 else w.d_k * es  # an 8-bit row carries its scale
        self.w, self.es = w, es
        kv_touch = self._decode_bytes((lens0 + CYCLE).tolist())
        n_rot = max(1, math.ceil(4 * L2_BYTES / kv_touch))
        cache_bytes = 2 * wb.B * wb.h_kv * n_max * row_bytes
        free = torch.cuda.mem_get_info(dev)[0]
        n_rot = int(max(1, min(n_rot, 64, (0.6 * free) // cache_bytes)))

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
        stream: a replay of `graph` (K steps recorded by capture()), or K eager calls."""
        ev_start = torch.cuda.Event(enable_timing=True)
        ev_end = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        # Keep the GPU busy (outside the timed region) while the host queues the
        # first steps, so that host launch latency does not leak into the timing.
        torch.cuda._sleep(int(5e7))
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
        graph, launches = h.capture(K)
        h.time_steps(K, world, graph)  # first replay: uploads the graph
    launches0 = api.launch_count()
    if sampler:
        sampler.mark(True)
    local_ms = h.time_steps(K, world, graph)
    if sampler:
        sampler.mark(False)
    if args.eager:
        launches = api.launch_count() - launches0
    del graph
    ms_per_step, tokens_per_s = replica_rate(local_ms, world, w.B, K)
    clocks = sampler.stop() if sampler else None

    # ---- end to end: pinned host inputs in, result out, every step
    # per step: q and the new rows (with their scales for an 8-bit cache)
    rows_d = [k_new, v_new] + ([h.k_new_scale, h.v_new_scale] if h.q8 else [])
    rows_h = [[t.cpu().pin_memory() for t in ts] for ts in rows_d]
    q_h = q.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    q_d = torch.empty_like(q)
    bufs = [torch.empty_like(ts[0]) for ts in rows_d]

    def e2e_step(i):
        c = i % CYCLE
        q_d.copy_(q_h, non_blocking=True)
        for b, hs in zip(bufs, rows_h):
            b.copy_(hs[c], non_blocking=True)
        step(i, q_d, *bufs)
        out_h.copy_(out, non_blocking=True)
        stream.synchronize()

    e2e_steps = max(1, min(K, 2000))
    for i in range(min(args.warmup, 8)):
        e2e_step(i)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    _, e2e_rate = replica_rate(1e3 * (time.perf_counter() - t0), world, w.B, e2e_steps)
    h2d = q.numel() * q.element_size() + sum(b.numel() * b.element_size() for b in bufs)
    d2h = out.numel() * out.element_size()

    if rank != 0:
        return
    # ---- accounting
    step_bytes = h.step_bytes()
    peak, peak_kind = peaks()
    achieved = step_bytes / (ms_per_step / 1e3) / 1e9
    traffic = recorded_traffic(w.name)
    bytes_str = f"{step_bytes / 1e6:.1f} MB per step"
    if w.B * w.h_kv * w.n * (w.d_k + w.d_v) * h.es < L2_BYTES:
        bytes_str += " (L2-resident)"

    cpu_v, cpu_sample, cpu_cores = oracle_step_sample(wb, args.cpu_seconds, 1)
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("f16 (8-bit codes, fp32 scales)" if h.q8
                  else "f32" if w.dtype == torch.float32 else "bf16"),
        "data": "synthetic", "config": workload_config(wb, n_rot, kv_touch),
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
                     "timing": "CUDA events around the K timed steps on the launching stream; "
                               "one kernel per step (two when splits are merged)",
                     "traffic": traffic, "algorithmic_bytes": step_bytes, "per": bytes_str},
        "cpu_baseline": {"value": cpu_v, "unit": "tokens/s", "cores": cpu_cores, "kind": "oracle",
                         "sample": cpu_sample},
        "e2e": {"value": e2e_rate, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "sync": "host waits for each step's result"},
        "gpu_launches": launches,
        "launch": ("eager: one C-ABI call per step" if args.eager else
                   "the K steps recorded once through the C-ABI into a CUDA graph, "
                   "replayed once inside the timed region"),
        "clocks": clocks,
    }
    print(json.dumps(line))


SWEEP_CONTEXTS = (1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072)
SWEEP_SHAPES = ("gqa_llama3_8b", "mqa_g32", "long_llama2_70b", "mha_fp32")


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
    ap.add_argument("--workload", default="mha_fp32", choices=sorted(W.WORKLOADS))
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
