"""The N > 1 path on CPU: world-size-2 gloo ranks, as bench.py runs them under
torchrun (one process per GPU; only a host barrier and a max over the ranks'
step times, no collective on the data path).

Covers the rank helper (barrier, max), the reference arm under torchrun (rank
0 alone prints one JSON line, the other rank exits 0 without work), and a
rank that dies before the barrier: the survivor must fail, not hang.
"""

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port, **extra):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    env.update({k: str(v) for k, v in extra.items()})
    return env


RANK_SCRIPT = r"""
import sys, time
sys.path.insert(0, {root!r})
import bench
d = bench.Dist()
mode = {mode!r}
if mode == "die" and d.rank == 1:
    import os
    os._exit(0)            # leaves without joining the barrier
try:
    d.barrier()
    v = d.max(1.5 + d.rank)
    print("RESULT", d.rank, d.world, v, flush=True)
    d.close()
except Exception as e:
    print("ERROR", d.rank, type(e).__name__, flush=True)
    sys.exit(3)
"""


def _run_ranks(mode, timeout_s=120, **extra):
    port = _free_port()
    script = RANK_SCRIPT.format(root=ROOT, mode=mode)
    procs = [subprocess.Popen([sys.executable, "-c", script], env=_env(r, 2, port, **extra),
                              stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
             for r in range(2)]
    outs = []
    for p in procs:
        try:
            out, _ = p.communicate(timeout=timeout_s)
        except subprocess.TimeoutExpired:
            p.kill()
            out, _ = p.communicate()
            out += "\nTIMEOUT"
        outs.append((p.returncode, out))
    return outs


def test_gloo_barrier_and_max_over_two_ranks():
    outs = _run_ranks("ok")
    for rank, (rc, out) in enumerate(outs):
        assert rc == 0, out
        line = [l for l in out.splitlines() if l.startswith("RESULT")][0].split()
        assert int(line[1]) == rank and int(line[2]) == 2
        assert float(line[3]) == 2.5                 # max over ranks of 1.5 + rank


def test_dead_rank_makes_the_survivor_fail_not_hang():
    outs = _run_ranks("die", timeout_s=90, BENCH_PG_TIMEOUT_S=10)
    rc0, out0 = outs[0]
    assert "TIMEOUT" not in out0, out0
    assert rc0 != 0 and "ERROR 0" in out0, out0


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3",
           "--workload", "1", "--ref-seconds", "3"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
