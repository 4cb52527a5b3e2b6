"""Host-side logic of the N-GPU bench path, on CPU with two gloo ranks.

The decode step shards by batch row with no collective on the data path: each
rank runs its own replica (its own seeded batch), and only the timing is
reduced -- the slowest rank's step time -- so the whole-job throughput is
units of all ranks / max time.
"""
import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    d = bench.init_dist(ws, "gloo")
    local_ms = 10.0 + 5.0 * rank                    # rank 1 is the slow one
    bench.barrier(d)
    ms = bench.max_over_ranks(d, local_ms, torch.device("cpu"))
    results[rank] = ms
    d.destroy_process_group()


def test_two_rank_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(world, port, results), nprocs=world, start_method="spawn", join=True)
    assert dict(results) == {0: 15.0, 1: 15.0}


def test_weak_scaling_value_counts_every_rank():
    import numpy as np

    import bench
    from decode_attention_self_gb300 import workloads as W

    w = W.make_workload(4)
    sb = bench.step_bytes(w)
    # per layer: valid K+V of every row, q and out, block-table entries; the step adds the sampler
    L = w.seq_len.astype(np.int64)
    expect_self = 4 * 16 * 64 * int(L.sum()) + 32 * 16 * 64 * (2 + 2) + 4 * int(((L + 15) // 16).sum())
    assert sb["self"] == expect_self
    assert sb["sampler"] == 32 * 9 * 1088 * 4 + 32 * 9 * 4
    assert sb["step"] == 24 * (sb["self"] + sb["cross"] + sb["append"]) + sb["sampler"]


def test_replicas_draw_distinct_batches():
    # each rank's replica is seeded by its rank: different data, same shapes
    from decode_attention_self_gb300 import workloads as W

    w = W.make_workload(1)
    a = W.make_step_inputs(w, 1000 * 0 + 0)[0]
    b = W.make_step_inputs(w, 1000 * 1 + 0)[0]
    assert a.shape == b.shape and not torch.equal(a, b)


def test_reference_arm_under_torchrun_prints_once():
    # Under torchrun the reference arm (the oracle on the host cores) runs on rank 0 alone; the other rank exits 0
    # without work, and exactly one JSON line comes out.
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(root, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # the same config object as the GPU arm prints for this workload, so that the two lines can be matched
    sys.path.insert(0, root)
    import bench
    from decode_attention_self_gb300 import workloads as W

    w = W.make_workload(1)
    sb = bench.step_bytes(w)
    assert d["config"] == bench.workload_config(w, sb, False, 2, bench.rotation_copies(sb["step"]))


def test_batch1_steps_rotate_enough_copies_to_leave_l2():
    # a step's data is used again only after >= 3x L2 of other data, or the figure says it is a warm-L2 one
    import bench
    from decode_attention_self_gb300 import workloads as W

    n = {i: bench.rotation_copies(bench.step_bytes(W.make_workload(i))["step"]) for i in range(1, 6)}
    assert n == {1: 1, 2: 3, 3: 2, 4: 1, 5: 1}
    for i in (2, 3):
        sb = bench.step_bytes(W.make_workload(i))["step"]
        assert n[i] * sb >= 3 * bench.L2_BYTES > (n[i] - 1) * sb
        assert "copies" in bench.l2_note(sb, n[i])
    assert "warm-L2" in bench.l2_note(bench.step_bytes(W.make_workload(1))["step"], 1)
    assert "larger than L2" in bench.l2_note(bench.step_bytes(W.make_workload(5))["step"], 1)
