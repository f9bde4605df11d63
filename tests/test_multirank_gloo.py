"""Multi-rank host logic of the benchmark on CPU: row shards cover every row
once with no overlap, and the timed region's maximum over ranks is what rank 0
reports.  Two gloo ranks on 127.0.0.1, spawned (no GPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, rows, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lo, hi = bench.shard_rows(rows, world, rank)
    fake_ms = 10.0 + 5.0 * rank                  # rank 1 is the slow one
    worst = bench.max_over_ranks(fake_ms, dist, "cpu")
    dist.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
        json.dump({"lo": lo, "hi": hi, "worst": worst}, fh)
    dist.destroy_process_group()


@pytest.mark.parametrize("rows", [4096, 4097, 1, 0])
def test_two_gloo_ranks(tmp_path, rows):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, rows, str(tmp_path)), nprocs=2,
                       join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    covered = [i for g in got for i in range(g["lo"], g["hi"])]
    assert covered == list(range(rows)), "shards must tile the rows in order"
    assert abs(got[0]["hi"] - got[0]["lo"] - (got[1]["hi"] - got[1]["lo"])) <= 1
    assert all(g["worst"] == 15.0 for g in got), "every rank sees the slowest rank's time"


def test_shard_rows_many_worlds():
    for world in (1, 2, 3, 8):
        for rows in (0, 1, 7, 4096, 65537):
            spans = [bench.shard_rows(rows, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == rows
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))


def test_reference_arm_contract():
    """--impl reference prints one JSON line with the oracle timed on the host."""
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                          "--warmup", "1", "--rows", "256", "--reference-seconds", "2"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_only_rank0_prints():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--rows", "64", "--reference-seconds", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert res.returncode == 0 and res.stdout.strip() == ""
