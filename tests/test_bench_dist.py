"""The benchmark's multi-rank path on CPU: two gloo ranks, no GPU.

Each rank runs an independent replica of the workload (the layer has no
exchange step between sequences or heads), so the only cross-rank traffic is
the timing reduction: the slowest rank's time sets the job's time, and the
job's throughput is the units of all ranks over that time.
"""
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    script = tmp_path / "rank.py"
    script.write_text(textwrap.dedent(f"""
        import os, sys
        sys.path.insert(0, {ROOT!r})
        import bench
        rank, world, local = bench._dist()
        assert world == 2 and rank in (0, 1)
        slowest = bench.aggregate_max(10.0 + 5.0 * rank, world)   # rank 1 is slower
        bench.barrier(world)
        print(f"rank {{rank}} max {{slowest}}")
        assert slowest == 15.0
    """))
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
    outs = [p.communicate(timeout=120)[0] for p in procs]
    for p, o in zip(procs, outs):
        assert p.returncode == 0, o
    assert "rank 0 max 15.0" in outs[0] and "rank 1 max 15.0" in outs[1]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    env_world = os.environ.get("WORLD_SIZE")
    assert env_world in (None, "1")
    assert bench.aggregate_max(3.5, 1) == 3.5


def test_reference_arm_on_non_zero_rank_prints_nothing(tmp_path):
    env = dict(os.environ, RANK="1", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
