"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

The layer runs as independent replicas (weak scaling), so the only cross-rank
steps are the barrier around the timed region and the max over ranks of the
elapsed time; the reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"), True)
    dist.barrier()
    with open(f"{out_path}.{rank}", "w") as fh:
        json.dump({"rank": rank, "max": slowest, "seed": bench.token_seed(rank)}, fh)
    dist.destroy_process_group()


def test_max_over_ranks_and_seeds_gloo(tmp_path):
    world = 2
    out = str(tmp_path / "r")
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    res = [json.load(open(f"{out}.{r}")) for r in range(world)]
    assert [r["max"] for r in res] == [15.0, 15.0]        # every rank sees the slowest time
    assert res[0]["seed"] == 0 and res[1]["seed"] != 0    # rank 0's batch is the parity-tested one


def test_single_rank_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    import torch

    assert bench.max_over_ranks(3.5, torch.device("cpu"), False) == 3.5


def test_reference_arm_runs_on_rank0_only():
    """Under torchrun, ranks other than 0 of the reference arm exit 0 silently."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--config", "tiny", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
