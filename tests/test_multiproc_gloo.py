"""The multi-process host paths on CPU, world size 2, gloo backend:

* the context-parallel exchange: each rank holds one segment's (M, S_zero) --
  computed here by the oracle -- all-gathers them and forms its initial state
  with cp.prefix_state; rank 1's must equal the oracle's state after segment 0;
* bench.py's rank plumbing: dist_setup from the torchrun environment, the
  barrier and the max-over-ranks of the timed region.
No GPU is used; the library is not loaded.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cp_worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import oracle
    from kimi_delta_attention_chunk_gb300 import cp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(61)
        T, H, K, V = 19, 2, 5, 3
        q, k, v = (rng.standard_normal((T, H, d)) for d in (K, K, V))
        g = np.maximum(-5.0, -np.logaddexp(0.0, rng.standard_normal((T, H, K))))
        b = rng.uniform(0.1, 1.0, (T, H))
        s0 = rng.standard_normal((H, K, V))
        cut = [0, 8, T]
        sl = slice(cut[rank], cut[rank + 1])
        _, s_zero = oracle.kda_forward(q[sl], k[sl], v[sl], g[sl], b[sl])
        M = torch.from_numpy(oracle.segment_transition(k[sl], g[sl], b[sl]))
        Sz = torch.from_numpy(s_zero[0])
        Ms = [torch.empty_like(M) for _ in range(world)]
        Ss = [torch.empty_like(Sz) for _ in range(world)]
        dist.all_gather(Ms, M)
        dist.all_gather(Ss, Sz)
        s_in = cp.prefix_state(Ms, Ss, torch.from_numpy(s0), rank, compose=lambda m, s, a: m @ s + a)
        _, s_ref = oracle.kda_forward(q[:cut[rank]], k[:cut[rank]], v[:cut[rank]], g[:cut[rank]],
                                      b[:cut[rank]], initial_state=s0[None])
        out[rank] = float(np.abs(s_in.numpy() - s_ref[0]).max())
    finally:
        dist.destroy_process_group()


def _bench_worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    try:
        bench.barrier(w)
        out[rank] = (w, r, bench.max_over_ranks(1.5 + rank, w))
    finally:
        dist.destroy_process_group()


def _run(worker):
    if torch.cuda.is_available():
        pytest.skip("a CPU-only test")
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        return dict(out)


def test_context_parallel_exchange_two_ranks():
    out = _run(_cp_worker)
    assert out[0] < 1e-12 and out[1] < 1e-12, out


def test_bench_rank_plumbing_two_ranks():
    out = _run(_bench_worker)
    assert out[0] == (2, 0, 2.5) and out[1] == (2, 1, 2.5), out
