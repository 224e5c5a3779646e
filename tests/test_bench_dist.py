"""bench.py's multi-process logic on CPU (gloo, world size 2) and its
reference arm.  No GPU: the ranks exchange timings exactly as the GPU run
does (barrier, then the maximum over ranks), which is all the replicas-only
multi-GPU path needs."""

import io
import json
import os
import socket
import contextlib

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    r, w, _ = bench.dist_setup()
    assert (r, w) == (rank, world)
    bench.barrier()
    got = bench.max_over_ranks(10.0 + 5.0 * rank)
    # the reference arm: rank 0 prints, the other ranks do no work
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(_ref_args(), r, w)
    out.put((rank, got, buf.getvalue()))
    dist.barrier()
    dist.destroy_process_group()


def _ref_args():
    class A:
        pass
    a = A()
    a.ref_sample, a.workers, a.warmup, a.steps = 4096, 2, 0, 1
    a.n, a.workload_desc = 1 << 31, "slab_2p31 (test)"
    return a


def test_two_gloo_ranks_take_the_max_and_rank0_prints():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    line = json.loads(res[0][2].strip())
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert res[1][2] == ""


def test_reference_arm_line_single_process():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(_ref_args(), 0, 1)
    line = json.loads(buf.getvalue())
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "cpu_baseline", "e2e", "config"):
        assert key in line
    assert line["metric"] == bench.METRIC and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
