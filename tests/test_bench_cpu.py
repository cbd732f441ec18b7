"""Host logic of bench.py on CPU: the reduction of every rank's time to the
slowest one over gloo ranks (world size 2, the plumbing the N-GPU bench uses
over NCCL), the whole-job throughput, and the reference arm's rank handling
(rank 0 alone prints its line; the other ranks exit 0 without work)."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = _bench().max_over_ranks(1.5 + rank, dist, "cpu")
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(repr(got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        assert float((tmp_path / f"rank{rank}.txt").read_text()) == 2.5


def test_max_over_ranks_single_process_is_identity():
    assert _bench().max_over_ranks(3.25, None, "cpu") == 3.25


def test_job_tops_counts_the_units_of_every_rank():
    b = _bench()
    one = b.job_tops(2.0, 1)
    assert b.job_tops(2.0, 4) == pytest.approx(4 * one)
    assert one == pytest.approx(3 * b.OPS_PER_PRODUCT / 2.0e-3 / 1e12)


def _reference(rank, world):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                           "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=900)


def test_reference_arm_prints_on_rank0_only():
    r1 = _reference(1, 2)
    assert r1.returncode == 0, r1.stderr
    assert r1.stdout.strip() == ""
    r0 = _reference(0, 2)
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
