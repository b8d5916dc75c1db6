"""The multi-rank host path on the CPU (gloo, world size 2): decode shards into
independent replicas, one per rank, with no collective on the data path; the only
exchange is the bench's whole-job figures (max time over ranks, summed work)."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reduce_rank(rank, world, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        b = _bench()
        # rank r took 1 + r ms and 5 - r ms, moved 10 (r + 1) bytes and launched r kernels
        got = b.reduce_over_ranks(world, "cpu", [1.0 + rank, 5.0 - rank], [10.0 * (rank + 1), float(rank)])
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_whole_job_figures_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_reduce_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert got[r] == ([2.0, 5.0], [30.0, 1.0]), got[r]


def test_one_rank_keeps_its_own_figures():
    b = _bench()
    assert b.reduce_over_ranks(1, "cpu", [3, 4.5], [7]) == ([3.0, 4.5], [7.0])


def test_ranks_draw_distinct_inputs_of_one_shape():
    """Weak scaling: every rank decodes its own batch of the same shape and length mix."""
    b = _bench()
    for name in ("llama3_8b_decode", "tiny"):
        w0, w1 = b.make_workload(name, 0), b.make_workload(name, 1)
        s0, s1 = w0.steps[0], w1.steps[0]
        assert s0.query.shape == s1.query.shape and w0.key_cache.shape[1:] == w1.key_cache.shape[1:]
        assert not torch.equal(s0.query, s1.query)
        assert b.make_workload(name, 1).steps[0].query.equal(s1.query)   # seeded


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """The reference arm launched as the multi-GPU bench is (two ranks, 127.0.0.1
    rendezvous): rank 0 alone times the oracle and prints one JSON line; the other rank
    exits 0 without work."""
    port = _free_port()
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2",
           "--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_clock_sampling_follows_the_rank_gpu(monkeypatch):
    b = _bench()
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "4,5,6,7")
    assert [b.smi_index(r) for r in range(4)] == [4, 5, 6, 7]
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "GPU-aaaa,GPU-bbbb")
    assert b.smi_index(1) == 1
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert b.smi_index(2) == 2
