"""Host logic of the benchmark's multi-rank path on CPU with gloo (world size 2):
environment parsing, max-over-ranks timing and the whole-job value.  Every rank
runs its own replica of the workload; there is no data exchange to test."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

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


def _reference_line(*extra):
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *extra],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


REFERENCE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                  "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "impl", "config",
                  "cpu_baseline", "e2e"}


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle timed on the host) on the default
    forward workload: one JSON line with the contract's keys, no device needed."""
    line = _reference_line("--steps", "1", "--warmup", "0")
    assert REFERENCE_KEYS <= set(line)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["workload"] == "gdn_fwd_bf16_b4h16t8192d128_h0"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_on_the_decode_workload():
    line = _reference_line("--workload", "gdn_decode_bf16_n256h16d128", "--steps", "2", "--warmup", "1")
    assert REFERENCE_KEYS <= set(line)
    assert line["config"]["workload"] == "gdn_decode_bf16_n256h16d128"
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]


def test_decode_inputs_are_seeded():
    sys.path.insert(0, ROOT)
    import bench
    a, b = bench.decode_inputs(), bench.decode_inputs()
    for x, y in zip(a, b):
        assert x.shape == y.shape and bool((x == y).all())
    N, H, d = bench.DECODE_SHAPE
    assert a[5].shape == (N, H, d, d) and a[0].shape == (N, H, d)


# ----------------------------------------------------------------------------- FLOP counts
class _Counted:
    """Wraps numpy so that every matrix product of the chunk form adds its
    2 m n k FLOPs to a counter (an independent tally of what the formulas claim)."""

    def __init__(self):
        import numpy as np

        self.n = 0
        outer = self

        class Arr(np.ndarray):
            def __matmul__(self, other):
                return outer._mm(np.asarray(self), np.asarray(other))

            def __rmatmul__(self, other):
                return outer._mm(np.asarray(other), np.asarray(self))

        self.Arr = Arr

    def _mm(self, a, b):
        import numpy as np
        self.n += 2 * a.shape[0] * a.shape[1] * b.shape[1]
        return np.matmul(a, b).view(self.Arr)

    def wrap(self, x):
        import numpy as np
        return np.asarray(x, dtype=np.float64).view(self.Arr)


def _chunkform():
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import chunkform
    return chunkform


def test_forward_flop_formula_counts_the_chunk_form_products():
    """bench.algorithmic_flops (forward) = the products the chunk form multiplies, per
    chunk (ragged tails included), times the heads, plus the solve's c^3 / 3 multiply-adds."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from chunkwise_delta_rule_02_gb300 import workloads as W
    cf = _chunkform()
    for C, T, dk, dv in ((64, 70, 8, 6), (16, 37, 4, 12)):
        w = W.Workload("fl", 2, 3, T, dk, "f32", True, False, 1, chunk=C)
        x = W.generate(w)
        x["v"] = x["v"][..., :1].expand(*x["v"].shape[:-1], dv).contiguous()
        cnt = _Counted()
        rng = np.random.default_rng(0)
        for _ in range(2 * 3):   # every (batch row, head)
            cf.fwd_seq(cnt.wrap(rng.normal(size=(T, dk))), cnt.wrap(rng.normal(size=(T, dk))),
                       cnt.wrap(rng.normal(size=(T, dv))), rng.random(T), -rng.random(T) / 16, None, C)
        solve = 3 * sum((2 * c ** 3) // 3 for c in bench.chunk_lengths(w, x))   # heads x chunks
        assert bench.algorithmic_flops(w, x) == cnt.n + solve


def test_backward_flop_formula_counts_the_backward_products():
    """bench.algorithmic_flops (backward) against the products of the chunk-form
    backward, less those it computes twice where the kernels compute them once: its
    second pass recomputes T (Gamma K), T V and W S_in, it forms Q S_in for the gate
    term (the kernels reuse dO S_in^T), and it applies dKK and dKK^T to K separately
    (the kernels add them first)."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from chunkwise_delta_rule_02_gb300 import workloads as W
    cf = _chunkform()
    C, T, dk, dv = 16, 37, 4, 6
    w = W.Workload("flb", 1, 1, T, dk, "f32", True, False, 1, chunk=C)
    x = W.generate(w)
    x["v"] = x["v"][..., :1].expand(*x["v"].shape[:-1], dv).contiguous()
    cnt = _Counted()
    rng = np.random.default_rng(1)
    cf.bwd_seq(cnt.wrap(rng.normal(size=(T, dk))), cnt.wrap(rng.normal(size=(T, dk))),
               cnt.wrap(rng.normal(size=(T, dv))), rng.random(T), -rng.random(T) / 16, None,
               cnt.wrap(rng.normal(size=(T, dv))), None, C)
    lens = bench.chunk_lengths(w, x)
    twice = sum(2 * (2 * c * c * dk + c * c * dv + 2 * c * dk * dv) for c in lens)
    solve = sum((2 * c ** 3) // 3 for c in lens)
    assert bench.algorithmic_flops(w, x, backward=True) == cnt.n - twice + solve


def test_roofline_takes_the_slower_bound():
    sys.path.insert(0, ROOT)
    import bench
    pk = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0, "bf16_tflops_sustained": 50.0}
    r = bench.roofline(1e9, 1e13, 1000.0, pk, "test", sustained=False)   # 1 ms of HBM, 100 ms of FLOPs
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.1) < 1e-12 and r["unit"] == "TFLOP/s"
    r = bench.roofline(1e9, 1e13, 1000.0, pk, "test", sustained=True)
    assert abs(r["frac"] - 0.2) < 1e-12 and r["peak"] == 50.0
    r = bench.roofline(1e11, 1e12, 1000.0, pk, "test", sustained=False)  # 100 ms of HBM, 10 ms of FLOPs
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.1) < 1e-12 and r["unit"] == "GB/s"


def test_forward_counts_of_the_headline_workload():
    """B4 H16 T8192 d128, C = 64: 1.83e5 FLOP and 1030 B per token-head (plus the
    states), so the forward is bound by HBM at the measured peaks."""
    sys.path.insert(0, ROOT)
    import bench
    from chunkwise_delta_rule_02_gb300 import workloads as W
    w = W.WORKLOADS["gdn_fwd_bf16_b4h16t8192d128_h0"]
    x = W.generate(w, T=128)   # two chunks per item: the count per token does not depend on T
    th = 4 * 16 * 128
    assert bench.algorithmic_flops(w, x) == th * (6 * 128 * 128 + 10 * 64 * 128) + 4 * 16 * 2 * (2 * 64 ** 3 // 3)
    assert bench.algorithmic_bytes(w, x) == th * 1030 + 2 * 4 * 16 * 128 * 128 * 4


def test_record_step_traffic_sums_one_launch_of_each_kernel(tmp_path):
    """The forward+backward step's traffic entry sums one launch each of the cooperative
    forward, the reverse scan and the per-chunk gradients, stamped with the hash of every
    kernel source; a capture with a kernel missing or repeated is refused."""
    import bench
    head = '"ID","Process ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'
    def row(i, k, m, v):
        return '"%d","1","%s","%s","byte","%s"\n' % (i, k, m, v)
    rows = [row(0, "k_other(int)", "dram__bytes_read.sum", "5")]
    for i, (k, rd, wr) in enumerate((("coop::k_coop_fwd<Cfg<64, 128>>(x)", "1,000", "24"),
                                     ("gdn::bsc::k_bscan_tc(x)", "300", "200"),
                                     ("gdn::btc::k_bwd_tc(x)", "2,000", "100")), start=1):
        rows += [row(i, k, "dram__bytes_read.sum", rd), row(i, k, "dram__bytes_write.sum", wr)]
    csv_path = tmp_path / "s.csv"
    csv_path.write_text("==PROF== noise\n" + head + "".join(rows))
    out = tmp_path / "traffic.json"
    e = bench.record_step_traffic(str(csv_path), "fb", "ncu ...", out=str(out))
    assert e["dram_read"] == 3300 and e["dram_write"] == 324 and e["dram_bytes_per_launch"] == 3624
    assert e["source_sha"] == bench.kernel_source_sha("step")
    bad = tmp_path / "b.csv"
    bad.write_text(head + "".join(rows[:5]))   # the gradients kernel missing
    with pytest.raises(SystemExit):
        bench.record_step_traffic(str(bad), "fb", "ncu ...", out=str(out))


def test_record_traffic_reads_one_launch_and_stamps_the_source(tmp_path):
    """The traffic entry is the read + write DRAM bytes of the named kernel's launch in
    an ncu CSV, stamped with the hash of its current sources (so that a changed kernel
    reads as unmeasured)."""
    import bench
    csv_path = tmp_path / "t.csv"
    head = '"ID","Process ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'
    rows = ['"0","1","k_other(int)","dram__bytes_read.sum","byte","5"\n',
            '"1","1","k_coop_fwd<(anonymous namespace)::Cfg<64, 128>>(CUtensorMap_st)","dram__bytes_read.sum","byte","1,000"\n',
            '"1","1","k_coop_fwd<(anonymous namespace)::Cfg<64, 128>>(CUtensorMap_st)","dram__bytes_write.sum","byte","24"\n']
    csv_path.write_text("==PROF== noise\n" + head + "".join(rows))
    out = tmp_path / "traffic.json"
    e = bench.record_traffic(str(csv_path), "k_coop_fwd", "wl", "ncu ...", out=str(out))
    assert e["dram_read"] == 1000 and e["dram_write"] == 24 and e["dram_bytes_per_launch"] == 1024
    assert e["source_sha"] == bench.kernel_source_sha("k_coop_fwd")
    import json
    assert json.load(open(out))["k_coop_fwd@wl"]["capture"] == "ncu ..."
