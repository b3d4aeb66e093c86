"""Host-side logic of bench.py without a GPU: replica aggregation over gloo ranks,
the reference arm's JSON line, and the profile/peak readers."""
import json
import os
import subprocess
import sys
from pathlib import Path


ROOT = Path(__file__).resolve().parent.parent


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    import bench
    bench.dist_init(world, "gloo")
    t = bench.max_over_ranks(1.0 + rank, world)
    s = bench.sum_over_ranks(10.0 * (rank + 1), world)
    bench.barrier(world)
    q.put((rank, t, s))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_replica_aggregation_over_gloo():
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, s in res:
        assert t == 2.0          # the job's time is the slowest rank's
        assert s == 30.0         # whole-job work is summed over replicas


def test_reference_arm_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                          "--steps", "200", "--warmup", "3", "--workload", "sd_point_mass_f32"],
                         capture_output=True, text=True, env=env, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "sd_point_mass_f32"


def test_reference_arm_nonzero_rank_is_silent():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                          "--steps", "10"], capture_output=True, text=True, env=env, timeout=300)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_peak_and_profile_readers():
    sys.path.insert(0, str(ROOT))
    import bench
    peak, kind = bench.hbm_peak()
    assert peak > 1000 and kind in ("measured", "fallback")
    assert len(bench.kernel_source_hash()) == 16
    assert bench.profiled_traffic("no_such_workload") is None


def test_kernel_hash_ignores_comments_but_not_code():
    sys.path.insert(0, str(ROOT))
    import bench
    src = "// header\nint f(int a) {  /* the sum\n of two */\n  return a + 1;  // one\n}\n\n"
    assert bench.code_only(src) == bench.code_only(src.replace("the sum", "a sum").replace("// one", ""))
    assert bench.code_only(src) != bench.code_only(src.replace("a + 1", "a + 2"))
    assert bench.code_only(src) == "int f(int a) {\n  return a + 1;\n}"


def test_graph_length_rounds_up_to_whole_multiples():
    sys.path.insert(0, str(ROOT))
    import bench
    assert [bench.graph_length(k) for k in (1, 7, 20, 30, 100, 150, 0)] == [100, 105, 100, 120, 100, 150, 100]
    for k in range(1, 260):
        g = bench.graph_length(k)
        assert g % k == 0 and g >= bench.MIN_GRAPH_STEPS and g - k < bench.MIN_GRAPH_STEPS
