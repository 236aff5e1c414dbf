"""bench.py's multi-rank plumbing on CPU: two gloo ranks, the job time is the
slowest rank's, the job throughput counts every rank's work, and the
reference arm runs on rank 0 only."""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(3.0 + 2.0 * rank)
        q.put((rank, ms, bench.job_throughput(6e12, ms, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=5) for _ in range(2))
    assert [o[1] for o in out] == [5.0, 5.0]             # both ranks see the slowest rank's time
    assert abs(out[0][2] - 6e12 * 2 / 5e-3 / 1e12) < 1e-9  # whole-job TFLOP/s


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5) == 7.5


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


@pytest.mark.parametrize("bad", [["--warmup", "2"]])
def test_bench_rejects_too_few_warmups(bad):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *bad],
                       capture_output=True, text=True, timeout=60)
    assert r.returncode != 0


def test_watchdog_prints_the_headline_and_exits_when_the_extras_stall():
    import json
    import subprocess
    import sys
    code = ("import sys, time; sys.path.insert(0, %r); import bench\n"
            "line = {'metric': 'm', 'value': 1.0}\n"
            "extra = {'adamw': {'gbs': 2.0}}\n"
            "bench.progress('RWKV block')\n"
            "dog = bench.Watchdog(0.3, line, extra)\n"
            "time.sleep(30)\n") % ROOT
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=20)
    assert r.returncode == 0
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["value"] == 1.0 and out["adamw"] == {"gbs": 2.0}
    assert out["stalled"]["phase"] == "RWKV block"
    assert "watchdog" in r.stderr


def test_watchdog_cancelled_in_time_stays_silent():
    import subprocess
    import sys
    code = ("import sys, time; sys.path.insert(0, %r); import bench\n"
            "dog = bench.Watchdog(0.5, {'value': 1.0})\n"
            "dog.cancel(); time.sleep(1.0); print('done')\n") % ROOT
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=20)
    assert r.returncode == 0 and r.stdout.strip() == "done"


def test_code_hash_ignores_comments_but_not_code(tmp_path):
    """The traffic figures stay keyed to the GEMM code: a comment edit keeps the
    key, a code edit changes it."""
    import bench
    a = tmp_path / "a.cu"
    a.write_text("// header\nint f(int x) {  // twice\n    return 2 * x; /* note */\n}\n")
    h0 = bench.code_hash([str(a)])
    a.write_text("// another header\n\nint f(int x) {\n    return 2 * x; /* other\n note */\n}\n")
    assert bench.code_hash([str(a)]) == h0
    a.write_text("int f(int x) {\n    return 3 * x;\n}\n")
    assert bench.code_hash([str(a)]) != h0
