"""The bench's multi-GPU host logic on CPU: two gloo ranks (127.0.0.1) run the replica
timing plumbing of bench.py -- the barrier and the max over ranks that makes the job's
time the slowest rank's -- and the reference arm stays silent on ranks other than 0."""
import multiprocessing as mp
import os
import socket
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update(CUDA_VISIBLE_DEVICES="", MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    ws, r, local = bench.dist_init()
    m = bench.max_over_ranks(10.0 * (rank + 1), ws)
    bench.barrier(ws)
    q.put((r, ws, dist.get_backend(), m))
    dist.destroy_process_group()


def test_replica_timing_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, *_ in results] == [0, 1]
    assert all(ws == 2 and backend == "gloo" and m == 20.0 for _, ws, backend, m in results)


def test_reference_arm_prints_only_on_rank_zero(capsys):
    sys.path.insert(0, ROOT)
    import bench
    from selective_state_space_141_b300 import inputs
    args = types.SimpleNamespace(steps=1, warmup=0, gpus=2)
    bench.run_reference(args, inputs.TINY, 2, rank=1)
    assert capsys.readouterr().out == ""


def test_reference_arm_json_line(capsys):
    """Rank 0 prints one JSON line with the bench contract's keys, the oracle as the timed
    program (cpu_baseline kind "oracle", its thread count and CPU), and an e2e object with no
    host-device bytes."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    from selective_state_space_141_b300 import inputs
    args = types.SimpleNamespace(steps=1, warmup=0, gpus=1)
    bench.run_reference(args, inputs.TINY, 1, rank=0)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["steps"] == 1
    assert line["value"] > 0 and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["cpu_model"]
    e = line["e2e"]
    assert e["value"] == line["value"] and e["unit"] == line["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
