"""Multi-rank host logic of the benchmark on CPU: row shards cover every row
once with no overlap, the timed region's maximum over ranks is what rank 0
reports, and the row-sharded mode hands each rank its own contiguous block of
one global batch (the byte offset and row count of its call) with the gammas
replicated.  Two gloo ranks on 127.0.0.1, spawned (no GPU)."""
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


def _shard_main(rank, world, port, rows, n, out_dir):
    """One rank of the row-sharded mode, on CPU: its plan, its block of the
    global workload (the gammas whole), and the oracle on that block."""
    import numpy as np
    import torch.distributed as dist

    import oracle
    from dual_epsilon_sandwich_gb300 import workloads as wl
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    plan = bench.shard_plan(rows, n, 4, world, rank)
    w = wl.sandwich_prefill(rows=rows, n=n)
    blk = bench.local_block(w.arrays, plan)
    e1, e2 = float(np.float32(w.eps)), float(np.float32(w.eps_pre))
    s, o = oracle.norm_residual_norm(*(blk[k].astype(np.float64) for k in
                                       ("block_out", "residual", "gamma_post", "gamma_pre")),
                                     e1, e2)
    plans = [None] * world
    dist.all_gather_object(plans, plan)
    base = w.arrays["block_out"].__array_interface__["data"][0]
    mine = blk["block_out"].__array_interface__["data"][0] if plan["rows"] else base + \
        plan["byte_offset"]
    np.save(os.path.join(out_dir, f"s{rank}.npy"), s)
    np.save(os.path.join(out_dir, f"o{rank}.npy"), o)
    with open(os.path.join(out_dir, f"plan{rank}.json"), "w") as fh:
        json.dump({"plan": plan, "plans": plans, "offset_in_global": mine - base,
                   "gamma_whole": blk["gamma_post"].shape[0] == n,
                   "block_shape": list(blk["residual"].shape)}, fh)
    dist.destroy_process_group()


@pytest.mark.parametrize("rows", [9, 2, 1])
def test_row_sharded_mode_two_gloo_ranks(tmp_path, rows):
    """Each rank's block starts at byte row0 * n * 4 of the global batch, holds
    `rows` rows and the whole gammas; the blocks tile the batch in order; and
    the per-rank results, put back in rank order, equal the result on the whole
    batch (rows are independent: sharding changes no value)."""
    import numpy as np

    import oracle
    from dual_epsilon_sandwich_gb300 import workloads as wl
    n = 64
    port = _free_port()
    mp.start_processes(_shard_main, args=(2, port, rows, n, str(tmp_path)), nprocs=2,
                       join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"plan{r}.json")) for r in range(2)]
    assert got[0]["plans"] == got[1]["plans"] == [g["plan"] for g in got]
    row = 0
    for g in got:
        p = g["plan"]
        assert p["row0"] == row and p["byte_offset"] == row * n * 4
        assert p["bytes"] == p["rows"] * n * 4 and g["offset_in_global"] == p["byte_offset"]
        assert g["block_shape"] == [p["rows"], n] and g["gamma_whole"]
        row += p["rows"]
    assert row == rows
    w = wl.sandwich_prefill(rows=rows, n=n)
    e1, e2 = float(np.float32(w.eps)), float(np.float32(w.eps_pre))
    s, o = oracle.norm_residual_norm(*(w.arrays[k].astype(np.float64) for k in
                                       ("block_out", "residual", "gamma_post", "gamma_pre")),
                                     e1, e2)
    s_cat = np.concatenate([np.load(tmp_path / f"s{r}.npy") for r in range(2)])
    o_cat = np.concatenate([np.load(tmp_path / f"o{r}.npy") for r in range(2)])
    assert np.array_equal(s_cat, s) and np.array_equal(o_cat, o)


def test_shard_plan_many_worlds():
    for world in (1, 2, 3, 8):
        for rows, n in ((0, 8), (1, 6656), (7, 5), (4096, 6656), (65537, 3)):
            plans = [bench.shard_plan(rows, n, 4, world, r) for r in range(world)]
            assert plans[0]["row0"] == 0
            assert sum(p["rows"] for p in plans) == rows
            for a, b in zip(plans, plans[1:]):
                assert b["row0"] == a["row0"] + a["rows"]
                assert b["byte_offset"] == a["byte_offset"] + a["bytes"]
            assert max(p["rows"] for p in plans) - min(p["rows"] for p in plans) <= 1


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
