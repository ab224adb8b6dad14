"""The N > 1 path of bench.py on CPU: two gloo ranks, as torchrun would start
them (RANK / WORLD_SIZE / MASTER_* in the environment, 127.0.0.1).  Decode
and prefill shard with no exchange, so the only collectives are the timing's
MAX all-reduce and the barriers; each rank times its own batch (a different
seed), and the whole-job value counts every rank's bytes over the slowest
rank's time.  The reference arm runs on rank 0 only."""
import multiprocessing
import os
import socket
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), GQA_BENCH_BACKEND="gloo")
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    from grouped_query_attention_09_b300 import workloads as W
    r, w, local = bench.dist_setup()
    total_ms = bench.max_over_ranks(10.0 + 5.0 * rank, w)  # rank 1 is the slow one
    bench.barrier(w)
    value = bench.job_value(1_000_000, w, 4, total_ms)
    # each rank's batch: the workload's seed plus the rank
    wl = W.WORKLOADS["tiny"]
    mine = W.DecodeWorkload(wl.name, wl.B, wl.Hq, wl.Hkv, wl.D, wl.Lmax, wl.len_lo, wl.len_hi, wl.seed + r)
    q = W.make_decode_inputs(mine)[0]
    args = types.SimpleNamespace(warmup=3, steps=1, ref_budget=0.01)
    ref_rc = bench.run_reference(args, r, w) if r != 0 else None  # non-zero ranks leave at once
    out.put((r, w, local, total_ms, value, float(q.float().sum()), ref_rc))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = multiprocessing.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, t0, v0, qs0, rc0), (r1, w1, l1, t1, v1, qs1, rc1) = res
    assert (r0, r1) == (0, 1) and w0 == w1 == 2 and (l0, l1) == (0, 1)
    assert t0 == t1 == 15.0                               # MAX over ranks
    assert v0 == v1 == pytest.approx(2 * 4 * 1_000_000 / 15e-3 / 1e9)  # both ranks' bytes, slowest time
    assert qs0 != qs1                                     # different batches per rank
    assert rc1 == 0                                       # the reference arm runs on rank 0 only
