"""The N > 1 path of bench.py on CPU with gloo, world size 2.

The optimizer step has no exchange step of its own (every data-parallel rank
applies the same update to its replica), so N GPUs run N independent replicas:
the only cross-rank operations are the barrier and the max over ranks of the
timed region.  These tests run those on two CPU processes."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        t = [0.25, 0.75][rank]
        m = bench.max_over_ranks(t)
        rate = bench.whole_job_rate(1000, 4, world, m)
        q.put((rank, m, rate, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_max_over_ranks_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, m, rate, env in res:
        assert m == 0.75                                 # every rank sees the slowest rank's time
        assert abs(rate - 1000 * 4 * 2 / 0.75 / 1e9) < 1e-15
        assert env[0] == rank and env[1] == 2


def test_reference_arm_under_torchrun_prints_once():
    """Under torchrun with 2 ranks, rank 0 alone times the oracle and prints one JSON line;
    the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.5"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["cpu_baseline"]["kind"] == "oracle"
    assert out["e2e"]["h2d_bytes_per_step"] == 0


# ---------------------------------------------------------------------------
# The sharded optimizer step on two CPU ranks ([ZRO] "The scheme" and "Operational
# sharp edges": each rank owns a slice of the flattened parameters, the squared
# norms are all-reduced before the root, and [MEG] section 6: the overflow flag is
# all-reduced so every rank steps or skips together).  Each rank runs the oracle's
# element-wise functions on its own slice only; the two all-reduces go through
# torch.distributed (gloo).  The slices come from the library's host-side
# tl_partition (no GPU involved) and must equal the oracle's cut points.
# ---------------------------------------------------------------------------

SHARD_NUMEL = [37, 4096, 5, 999, 2048, 1, 3000]
SHARD_STEPS = 5
SHARD_OVERFLOW = (3, 1, sum(SHARD_NUMEL) - 7)   # (step, micro-batch, element): in rank 1's slice


def _shard_inputs(step, P, S):
    import numpy as np
    import oracle
    rng = np.random.default_rng([39, 17, step])
    grads = [oracle.recast(rng.standard_normal(P).astype(np.float32) * 0.05 * S, "f16") for _ in range(3)]
    if step == SHARD_OVERFLOW[0]:
        grads[SHARD_OVERFLOW[1]][SHARD_OVERFLOW[2]] = 0x7C00
    return grads


def _shard_worker(rank, world, port, q):
    import ctypes
    import numpy as np
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import oracle
    import loss_scaled_adamw_gb300 as tl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lib = oracle.load()
        P = sum(SHARD_NUMEL)
        # this rank's slice: the library's pieces, checked against the oracle's cut points
        pieces = tl.tl_partition(SHARD_NUMEL, world, rank, 16)
        starts = [sum(SHARD_NUMEL[:t]) + s for t, s, _ in pieces]
        lo, hi = starts[0], starts[-1] + pieces[-1][2]
        assert all(a + n == b for a, (_, _, n), b in zip(starts, pieces, starts[1:]))   # contiguous
        b = oracle.partition_bounds(P, world, 16)
        assert (lo, hi) == (int(b[rank]), int(b[rank + 1]))
        n = hi - lo
        rng = np.random.default_rng(5)
        master = (rng.standard_normal(P).astype(np.float32) * 0.02)[lo:hi].copy()
        w, m, v = master, np.zeros(n, np.float32), np.zeros(n, np.float32)
        p = oracle.recast(w, "f16")
        acc = np.empty(n, np.float32)
        state = oracle.State(2.0 ** 10, 0, 0, 1.0, 1.0)
        cfg = oracle.ScalerCfg(1, 2.0, 0.5, 2, 1.0, 2.0 ** 127)
        hp = oracle.AdamWHP(1e-3, 0.9, 0.95, 1e-8, 0.1)
        P_ = lambda a: a.ctypes.data_as(ctypes.c_void_p)
        counts = [3, 1, 2]
        log = []
        for step in range(1, SHARD_STEPS + 1):
            grads = _shard_inputs(step, P, state.S)
            for i, g in enumerate(grads):
                gi = np.ascontiguousarray(g[lo:hi])
                lib.tlo_accumulate(P_(acc), P_(gi), oracle.DT_F16, n, lib.tlo_microbatch_weight(counts[i], 6),
                                   1 if i == 0 else 0)
            flag = lib.tlo_unscale_check(P_(acc), n, state.S)
            local = lib.tlo_sumsq(P_(acc), n)
            s = torch.tensor([local], dtype=torch.float64)
            f = torch.tensor([flag], dtype=torch.int32)
            dist.all_reduce(s, op=dist.ReduceOp.SUM)
            dist.all_reduce(f, op=dist.ReduceOp.MAX)
            sumsq, found = float(s.item()), int(f.item())
            if not found and not np.isfinite(sumsq):
                found = 1
            b1n = state.b1p * float(np.float32(hp.beta1))
            b2n = state.b2p * float(np.float32(hp.beta2))
            norm = coef = None
            if not found:
                norm = lib.tlo_norm_from_sumsq(sumsq)
                coef = lib.tlo_clip_coef(norm, 1.0)
                sc = lib.tlo_adamw_prepare(ctypes.byref(hp), b1n, b2n)
                lib.tlo_adamw_recast(P_(w), P_(m), P_(v), P_(p), oracle.DT_F16, P_(acc), n, coef, ctypes.byref(sc))
            lib.tlo_scaler_update(ctypes.byref(state), ctypes.byref(cfg), found, b1n, b2n)
            log.append((step, found, norm, coef, state.S, state.t, flag))
        # gather every rank's slice on every rank
        out = {}
        for name, a in (("w", w), ("m", m), ("v", v), ("p", p.astype(np.int32))):
            t = torch.from_numpy(np.ascontiguousarray(a))
            sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
            dist.all_gather(sizes, torch.tensor([t.numel()], dtype=torch.int64))
            big = max(int(sz.item()) for sz in sizes)      # gloo gathers equal sizes: pad, then trim
            padded = torch.zeros(big, dtype=t.dtype)
            padded[:t.numel()] = t
            parts = [torch.zeros(big, dtype=t.dtype) for _ in sizes]
            dist.all_gather(parts, padded)
            out[name] = torch.cat([x[:int(sz.item())] for x, sz in zip(parts, sizes)]).numpy()
        out["p"] = out["p"].astype(np.uint16)
        q.put((rank, log, out if rank == 0 else None))
    finally:
        dist.destroy_process_group()


def test_sharded_step_on_two_gloo_ranks():
    import numpy as np
    import oracle
    from loss_scaled_adamw_gb300 import _build
    _build.build()          # tl_partition lives in the library (host code only here)
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    import queue
    import time
    got, t0 = [], time.time()
    while len(got) < 2:
        try:
            got.append(q.get(timeout=2))
        except queue.Empty:
            assert not any(p.exitcode not in (None, 0) for p in procs), "a rank failed"
            assert time.time() - t0 < 300, "ranks did not finish"
    res = sorted(got, key=lambda x: x[0])
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    logs = [r[1] for r in res]
    # both ranks took the same decisions and moved S the same way
    assert [e[:6] for e in logs[0]] == [e[:6] for e in logs[1]]
    assert [e[1] for e in logs[0]] == [0, 0, 1, 0, 0]
    # the overflow was only in rank 1's slice: rank 0's local flag stayed clear
    assert logs[0][2][6] == 0 and logs[1][2][6] == 1
    # the gathered state equals the unsharded oracle's, and the sharded statement's
    P = sum(SHARD_NUMEL)
    rng = np.random.default_rng(5)
    master = rng.standard_normal(P).astype(np.float32) * 0.02
    for shards in (None, (2, 16)):
        o = oracle.Oracle(master, oracle.recast(master, "f16"), "f16", "f16", scaler_enabled=True,
                          init_scale=2.0 ** 10, interval=2)
        for step in range(1, SHARD_STEPS + 1):
            r = o.step(_shard_inputs(step, P, o.state.S), [3, 1, 2], 1.0, shards=shards)
            e = logs[0][step - 1]
            assert r.skipped == e[1] and o.state.S == e[4] and o.state.t == e[5]
            if not r.skipped:
                assert r.norm == e[2] and r.coef == e[3]
        got = res[0][2]
        for f in ("w", "m", "v", "p"):
            assert np.array_equal(got[f], getattr(o, f)), (shards, f)
