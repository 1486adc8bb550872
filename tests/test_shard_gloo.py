"""The sharded decode's exchange step with two gloo ranks on the CPU.

Each rank holds a disjoint set of cached rows of every sequence.  Its partial
(normalised output and natural-log log-sum-exp) comes from the oracle here,
since the CPU has no kernels; ``shard.gather_partials`` (the product's
all-gather into local tensors) collects them, and the oracle's log-sum-exp
merge of the gathered parts must equal the oracle's decode over all rows.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    import torch.distributed as dist

    import oracle
    from decode_attention_kv_split_gb300 import shard, workloads as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        o = oracle.get()
        w = W.custom(B=3, h_q=8, h_kv=2, d_k=64, n=90, n_max=90, dtype=torch.float32)
        K, V = W.cache(w, 5)
        q = W.query(w, 5).numpy()
        lens = np.array([90, 41, 0], dtype=np.int32)
        # rank r holds rows l with l % world == r (any disjoint cut works)
        mine = [np.arange(r, int(n), world) for r, n in zip([rank] * w.B, lens)]
        width = max(1, max(len(m) for m in mine))
        Ks = np.zeros((w.B, w.h_kv, width, w.d_k), dtype=np.float32)
        Vs = np.zeros_like(Ks)
        for b, rows in enumerate(mine):
            Ks[b, :, :len(rows)] = K.numpy()[b][:, rows]
            Vs[b, :, :len(rows)] = V.numpy()[b][:, rows]
        my_o, my_l = o.decode(q, Ks, Vs, np.array([len(m) for m in mine], dtype=np.int32),
                              w.scale)
        o_parts, l_parts = shard.gather_partials(torch.from_numpy(my_o).float(),
                                                 torch.from_numpy(my_l).float())
        assert o_parts.shape == (world, w.B, w.h_q, w.d_v) and l_parts.shape == (world, w.B, w.h_q)
        # part `rank` is this rank's own partial
        assert torch.equal(o_parts[rank], torch.from_numpy(my_o).float())
        merged = np.zeros((w.B, w.h_q, w.d_v))
        merged_l = np.zeros((w.B, w.h_q))
        for b in range(w.B):
            for h in range(w.h_q):
                merged[b, h], merged_l[b, h] = o.lse_combine(o_parts[:, b, h].double().numpy(),
                                                             l_parts[:, b, h].double().numpy())
        want, want_l = o.decode(q, K.numpy(), V.numpy(), lens, w.scale)
        err = float(np.max(np.abs(merged - want)))
        fin = np.isfinite(want_l)
        lerr = float(np.max(np.abs(merged_l[fin] - want_l[fin])))
        empty_ok = bool(np.all(np.isneginf(merged_l[~fin])) and np.all(merged[2] == 0))
        results.put((rank, err, lerr, empty_ok))
    finally:
        dist.destroy_process_group()


def test_gather_then_merge_equals_unsharded_decode():
    world = 2
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(results.get(timeout=5) for _ in range(world))
    for rank, err, lerr, empty_ok in got:
        # the partials travel as float32, so the merge matches to float32 rounding
        assert err < 1e-6, (rank, err)
        assert lerr < 1e-5, (rank, lerr)
        assert empty_ok
