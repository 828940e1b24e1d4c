"""The bench's multi-rank path on CPU (gloo, world size 2), and its reference arm.

The GEMM does not shard in this library: `bench.py --gpus N` runs N
independent replicas and only needs a barrier and a max over ranks of the
timed region.  Those steps are exercised here with the gloo backend, as are
the whole-job throughput formula and the `--impl reference` arm (the CPU
oracle timed on a bounded sample), none of which needs a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        pass

    w, r, local, pg = bench.dist_setup(Args())
    try:
        assert (w, r) == (world, rank) and pg is not None
        bench.barrier(pg)
        slowest = bench.max_over_ranks(pg, 10.0 + rank, "cpu")  # rank 1 is slower
        out[rank] = (slowest, bench.whole_job_tflops(1_000_000_000, 100, w, slowest))
    finally:
        pg.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_region():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 11.0
    # 2 ranks x 100 steps x 1 GFLOP over 11 ms
    assert abs(res[0][1] - 2 * 100 * 1e9 / 11e-3 / 1e12) < 1e-9


def test_whole_job_formula_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert abs(bench.whole_job_tflops(2 * 4096 ** 3, 10, 1, 1.0) - 2 * 4096 ** 3 * 10 / 1e-3 / 1e12) < 1e-9


def test_reference_arm_prints_one_json_line():
    """`bench.py --impl reference` times the oracle on the host: it needs no
    GPU and must print exactly one JSON line with the arm's fields."""
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "int512", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["config"]["workload"] == "int512"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_bench_shape_and_plan_options_parse():
    """--shape takes the workload's inputs at another size (and drops the other
    configurations); --plan-options sets hgemm_options_t fields by name and
    refuses unknown ones."""
    sys.path.insert(0, ROOT)
    import bench
    from tensor_core_dense_swizzled_gb300 import inputs
    w = inputs.WORKLOADS["square4096"]
    old = sys.argv
    try:
        sys.argv = ["bench.py", "--shape", "512,256,128", "--plan-options", "cta_pair=2,group_m=8"]
        args = bench.parse()
        opt = bench.plan_options(args, w)
        assert (opt.cta_pair, opt.group_m, opt.trans_b) == (2, 8, 0)
        assert args.shape == "512,256,128"
        sys.argv = ["bench.py", "--plan-options", "no_such_field=1"]
        args = bench.parse()
        try:
            bench.plan_options(args, w)
            raise AssertionError("an unknown field was accepted")
        except SystemExit:
            pass
    finally:
        sys.argv = old
