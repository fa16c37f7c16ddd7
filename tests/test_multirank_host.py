"""Multi-rank host logic of the benchmark on CPU: two gloo ranks.

The decode step shards with no exchange: every rank runs its own batch of
the workload at the full per-GPU size (weak scaling), and the only
collectives are the barrier around the timed region and the max over ranks
of its duration.  These tests run that logic as two processes on CPU and
check (1) the max-over-ranks reduction and the whole-job throughput formula,
(2) that the ranks draw disjoint synthetic batches of equal shape, and
(3) that the reference arm runs on rank 0 only.
"""
import contextlib
import io
import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(WORLD), LOCAL_RANK=str(rank))


class _Args:
    impl = "ours"
    workload = "whisper_large_b32"
    layers = 1
    steps = 2
    warmup = 3


def _rank_main(rank, port, outdir):
    _env(rank, port)
    import numpy as np
    import torch.distributed as dist
    import bench
    from kv_cache_decode_asr_gb300 import synthetic as syn

    world, r, _ = bench.dist_setup(_Args)
    assert (world, r) == (WORLD, rank)
    cpu = torch.device("cpu")
    # each rank times a different region; the job takes the slowest
    ms_total = 10.0 * (rank + 1)
    ms_step, value = bench.job_throughput(ms_total, 4, 32, world, cpu)
    bench.barrier(world)
    # this rank's synthetic batch: first tensor of the workload, host draw
    base = bench.rank_seed_base("whisper_large_b32", rank)
    q = syn.host_normal_f32((32, 1280), syn.seed_for(base, 1))
    res = {"ms_step": ms_step, "value": value, "base": base,
           "q_shape": list(q.shape), "q_sum": float(np.float64(q).sum())}
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)
    dist.destroy_process_group()


def _reference_main(rank, port, outdir):
    _env(rank, port)
    import torch.distributed as dist
    import bench

    class A(_Args):
        impl = "reference"

    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(A)
    with open(os.path.join(outdir, f"ref{rank}.txt"), "w") as f:
        f.write(buf.getvalue())
    if dist.is_initialized():
        dist.destroy_process_group()


def test_two_ranks_max_reduce_and_disjoint_batches(tmp_path):
    mp.start_processes(_rank_main, args=(_free_port(), str(tmp_path)), nprocs=WORLD,
                       start_method="spawn")
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(WORLD)]
    # both ranks see the slowest rank's 20 ms over 4 steps = 5 ms per step
    for x in r:
        assert x["ms_step"] == pytest.approx(5.0)
        assert x["value"] == pytest.approx(32 * WORLD / 5e-3)
    # equal per-rank shapes (weak scaling), different seeds and values
    assert r[0]["q_shape"] == r[1]["q_shape"] == [32, 1280]
    assert r[0]["base"] != r[1]["base"]
    assert r[0]["q_sum"] != r[1]["q_sum"]


def test_reference_arm_runs_on_rank_zero_only(tmp_path):
    mp.start_processes(_reference_main, args=(_free_port(), str(tmp_path)), nprocs=WORLD,
                       start_method="spawn")
    out0 = (tmp_path / "ref0.txt").read_text().strip().splitlines()
    out1 = (tmp_path / "ref1.txt").read_text()
    assert out1 == ""
    assert len(out0) == 1
    line = json.loads(out0[0])
    assert line["impl"] == "reference"
