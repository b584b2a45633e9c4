"""Host logic of the benchmark's multi-rank path on CPU with gloo (world size 2):
environment parsing, max-over-ranks timing and the whole-job value.  Every rank
runs its own replica of the workload; there is no data exchange to test."""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    env = bench.dist_env()
    ms = bench.max_over_ranks(2.0 + 3.0 * rank, dist, "cpu")
    q.put((rank, env, ms, bench.whole_job_value(1000, env[1], ms)))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, ms, value in res:
        assert env == (rank, 2, rank)
        assert ms == 5.0                       # the slowest rank's time on every rank
        assert abs(value - 2000 / 0.005) < 1e-6


def test_single_rank_defaults():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_value(524288 // 16, 1, 1.0) == 32768 * 1000.0


def test_cpu_baseline_counts_the_tokens_it_runs():
    """The oracle leg gathers its items into one call; the tokens it reports are the
    items' tokens divided by the heads (whole tokens), for fixed and packed input."""
    sys.path.insert(0, ROOT)
    import bench
    from chunkwise_delta_rule_02_gb300 import workloads as W
    w = W.Workload("cb", 2, 3, 40, 8, "bf16", True, True, 1)
    x = W.generate(w)
    secs, tok = bench.oracle_sample_fwd(x, w, bench.sample_items(x, 4), 2)
    assert secs > 0 and abs(tok - 40 * 4 / 3) < 1e-9
    wv = W.Workload("cbv", 1, 2, 0, 8, "bf16", True, True, 2, varlen_total=1, varlen_n=1)
    xv = W.generate(wv, lengths=[3, 0, 50])
    secs, tok = bench.oracle_sample_fwd(xv, wv, bench.sample_items(xv, 100), 2)
    assert secs > 0 and abs(tok - 53) < 1e-9
    cb = bench.cpu_baseline(x, w)
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
