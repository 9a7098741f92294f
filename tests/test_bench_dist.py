"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2): the
max-over-ranks timing reduction, and the reference arm printing exactly one JSON line
from rank 0 while the other rank exits cleanly."""
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


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(1.5 + 2.0 * rank, dist)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 3.5, 1: 3.5}


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.25, None) == 2.25


def test_reference_arm_two_ranks_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "vsa_tiny",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_backward_cpu_sample_reports_the_threads_it_used():
    # the oracle backward runs key/value heads in parallel: the sample spans as many heads
    # as the oracle has threads (at most H), and reports that count as its cores
    import bench
    from block_sparse_attention_vsa_gb300 import workloads
    from oracle import oracle as orc
    w = workloads.make_random_vsa(1, 3, 8 * 64, 128, 64, 4, seed=5, n_lo=1)
    pairs, seconds, n_blocks, threads, heads = bench.oracle_bwd_sample(w, 0.01)
    assert heads == threads == min(orc.num_threads(orc.load()), 3)
    assert n_blocks >= 1 and seconds > 0.0
    # the attended pairs of those heads' first n_blocks query blocks
    mask = orc.lut_to_blockmask(w.q2k_idx[:1, :heads, :n_blocks], w.q2k_num[:1, :heads, :n_blocks],
                                w.nbk)
    assert pairs == int(mask.sum()) * 64 * 64
