"""Host-side logic of the benchmark (no GPU): the multi-rank path with two
gloo ranks on the CPU, the whole-job aggregate, the L2 policy and the
reference arm's output contract."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    w, r, lr, pg = bench.dist_setup(world)
    bench.barrier(pg)
    slowest = bench.max_over_ranks(pg, 10.0 + 5.0 * rank)    # rank 1 is slower
    value = bench.aggregate_tflops(w, 2.0e12, 4, slowest)
    bench.barrier(pg)
    pg.destroy_process_group()
    q.put((rank, w, r, slowest, value))


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, w, r, slowest, value in out:
        assert (w, r) == (world, rank)
        assert slowest == 15.0                        # max over ranks
        # 2 ranks x 4 steps x 2 TFLOP in 15 ms
        assert value == pytest.approx(2 * 4 * 2.0 / 15e-3)


def test_aggregate_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_tflops(1, 1e12, 10, 1000.0) == pytest.approx(10.0)


def test_l2_policy_by_input_size():
    sys.path.insert(0, ROOT)
    import bench
    from tiled_mma_atom_gb300 import inputs
    W = inputs.WORKLOADS
    assert bench.l2_policy(W["bf16_4096"])[0] is True
    assert bench.l2_policy(W["mxfp4_8192"])[0] is True
    assert bench.l2_policy(W["skinny_16x28672x8192"])[0] is False
    assert bench.input_bytes(W["skinny_16x28672x8192"]) == (16 + 28672) * 8192 * 2


def test_reference_arm_prints_one_line_on_cpu():
    """--impl reference runs the CPU oracle only and prints one JSON line."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--workload", "fp32_128"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_config_block_is_last_and_fits_a_short_tail():
    """The five configurations' compact entries close the JSON line, so a
    reader that keeps only the last 1,500 characters still sees C1-C5 with
    their oracle timings and their warm (back-to-back) times.  Built from realistic values through the same
    helpers bench.py uses."""
    sys.path.insert(0, ROOT)
    import bench
    from tiled_mma_atom_gb300 import inputs
    peaks = {"hbm_gbs": 6776.6, "bf16_tflops": 1905.4, "bf16_tflops_sustained": 1719.9}
    configs = {}
    for i, name in enumerate(bench.CONFIGS):
        w = inputs.WORKLOADS[name]
        ms = [0.0123456789, 0.0823456789, 0.1823456789]
        rl = bench.roofline(w, sum(ms) / 3, peaks, "measured", {})
        configs[f"C{i + 1}_{name}"] = bench.config_entry(w, ms, rl, (0.0461234, 2.98765, 935, 16), 0.0712345678)
    line = {"metric": bench.METRIC, "value": 1613.6, "workloads": {"x": {"tflops": 1.0}}, "configs": configs}
    text = json.dumps(line)
    tail = text[-1500:]
    for i, name in enumerate(bench.CONFIGS):
        assert f'"C{i + 1}_{name}"' in tail
    assert list(json.loads(text))[-1] == "configs"
    c5 = configs["C5_mxfp4_8192"]
    assert c5["bound"] == "tensor" and c5["kernel"] == "mxfp4_pair_kernel"
    assert c5["cpu"]["cores"] == 16 and c5["cpu"]["rows"] == "935/8192"
    assert configs["C4_skinny_16x28672x8192"]["unit"] == "GB/s"
    assert c5["ms_warm"] == 0.07123 and c5["ms"] == 0.09235
    assert bench.sig(0.0823456789) == 0.08235 and bench.sig(1613.61) == 1614.0
