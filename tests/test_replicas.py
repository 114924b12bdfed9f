"""The N > 1 bench harness on CPU: world-size-2 gloo ranks launched the way the driver launches
bench.py (torch.distributed.run, 127.0.0.1). Independent replicas: no data-path collective, only
a barrier and a max-over-ranks reduction of the timings; rank 0 alone prints."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, env=None, timeout=180):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    e = dict(os.environ)
    e.update(env or {})
    e.setdefault("OMP_NUM_THREADS", "1")
    return subprocess.run(cmd, cwd=ROOT, env=e, capture_output=True, text=True, timeout=timeout)


def test_max_over_ranks_and_whole_job_rate(tmp_path):
    out = str(tmp_path / "rank")
    p = _torchrun([os.path.join("tests", "replica_worker.py")], env={"REPLICA_OUT": out})
    assert p.returncode == 0, p.stderr[-2000:]
    res = [json.load(open(f"{out}.{r}")) for r in range(2)]
    for r in res:
        assert r["world"] == 2
        assert r["ms"] == 11.0 and r["e2e"] == 23.0          # the slowest rank's times
        assert abs(r["value"] - 2 * 5 * 1024 / 0.011) < 1e-6  # both ranks' tokens / max time


def test_reference_arm_prints_once_under_torchrun():
    p = _torchrun(["bench.py", "--impl", "reference", "--config", "c1", "--gpus", "2",
                   "--steps", "1", "--warmup", "0"])
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
