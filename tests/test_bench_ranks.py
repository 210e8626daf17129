"""The multi-replica path of bench.py on CPU: world-size-2 gloo ranks check
that the timed region is the slowest rank's, that the whole-job value counts
every replica's work, that replicas draw different inputs, and that under a
launcher only rank 0 of the reference arm does any work."""

import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        own = 1.0 + 2.5 * rank                       # rank 1 is the slow one
        ms = bench.slowest_rank_ms(own, world)
        dist.barrier()
        q.put((rank, ms, bench.whole_job_tflops(world, 3.0e9, ms), bench.replica_seed(rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_the_slowest_and_count_both_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, v0, s0), (r1, ms1, v1, s1) = got
    assert (r0, r1) == (0, 1)
    assert ms0 == ms1 == 3.5                          # both ranks report the slowest rank's time
    assert v0 == v1 == 2 * 3.0e9 / 3.5e-3 / 1e12      # two replicas' work over that time
    assert s0 != s1                                   # each replica draws its own inputs


def test_single_rank_needs_no_process_group():
    assert bench.slowest_rank_ms(2.0, 1) == 2.0
    assert bench.whole_job_tflops(1, 1.0e12, 1000.0) == 1.0


def test_replica_inputs_differ_but_do_the_same_work():
    from paged_decode_attention_fp8_gb300 import synthetic as syn
    lens = syn.uniform_seqlens(2, 4, 64, 200)
    a = syn.mla_inputs(bench.replica_seed(0), 4, 2, 64, lens, causal=True)
    b = syn.mla_inputs(bench.replica_seed(1), 4, 2, 64, lens, causal=True)
    assert a.seqlens.tolist() == b.seqlens.tolist()
    assert not bool((a.q == b.q).all())


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
