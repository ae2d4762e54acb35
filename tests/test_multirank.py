"""The N > 1 host logic of bench.py on CPU: two gloo ranks (127.0.0.1).

bench.py runs one independent replica per rank (sequences shard across
ranks, no collective on the data path); the only cross-rank steps are the
barriers around the timed region and the maximum of the step time.  These
tests run those helpers in two processes and check the whole-job
aggregation, and that the reference arm's non-zero ranks exit without work."""
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    import synth
    import torch.distributed as dist
    try:
        n = bench.dist_init("gloo")
        bench.dist_barrier()
        # per-rank step times; the job's time is the slowest rank's
        t = bench.dist_max(1.0 + 3.0 * rank)
        value = bench.aggregate_throughput(100, n, t)
        # each rank draws its own sequences (independent shards)
        tok = synth.tokens(synth.SMALL, 2, 16, seed=1000 + rank)
        bench.dist_barrier()
        q.put((rank, n, t, value, tok.tolist()))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_ranks_time_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, n, t, value, _ in res:
        assert n == 2
        assert t == 4.0                       # max over ranks of 1 + 3 rank
        assert value == 100 * 2 / 4.0         # every rank's tokens over the slowest time
    assert res[0][4] != res[1][4]             # ranks hold different sequences


def test_single_process_helpers_need_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(2.5) == 2.5
    bench.dist_barrier()                      # no-op without a process group
    assert bench.aggregate_throughput(10, 1, 2.0) == 5.0


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "{" not in r.stdout                # only rank 0 prints the JSON line
