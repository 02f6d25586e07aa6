"""The N > 1 path of bench.py on CPU: two gloo ranks, launched like torchrun
would (RANK / WORLD_SIZE / MASTER_* in the environment).  On GPUs each rank
is an independent replica of the round (no collective on the data path);
what crosses ranks is only the start/stop barrier, the max-over-ranks of the
timed interval, and rank 0 printing the line."""
import contextlib
import io
import json
import os
import queue
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(ws),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    got_ws, got_rank, _ = bench.dist_setup()
    assert dist.get_backend() == "gloo"
    bench.barrier(got_ws)
    # every rank reports a different elapsed time; all must agree on the max
    mx = bench.reduce_max(10.0 * (rank + 1), got_ws)
    rate = bench.whole_job_rate(steps=50, ws=got_ws, max_ms=mx)
    # the reference arm: rank 0 alone runs and prints, the others exit quietly
    buf = io.StringIO()
    sys.argv = ["bench.py", "--impl", "reference", "--gpus", str(ws), "--steps", "1", "--warmup", "0",
                "--workload", "tiny"]
    with contextlib.redirect_stdout(buf):
        bench.main()
    bench.barrier(got_ws)
    dist.destroy_process_group()
    q.put((got_rank, got_ws, mx, rate, buf.getvalue()))


@pytest.mark.timeout(300)
def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = []
    while len(res) < len(ps):
        try:
            res.append(q.get(timeout=5))
        except queue.Empty:
            dead = [p.exitcode for p in ps if p.exitcode not in (None, 0)]
            assert not dead, f"a rank failed with exit code {dead}"
    res.sort()
    for p in ps:
        p.join(60)
        assert p.exitcode == 0
    (r0, ws0, mx0, rate0, out0), (r1, ws1, mx1, rate1, out1) = res
    assert (r0, r1, ws0, ws1) == (0, 1, 2, 2)
    assert mx0 == mx1 == 20.0
    # whole-job throughput: both ranks' units over the slowest rank's time
    assert rate0 == rate1 == pytest.approx(2 * 50 / 0.020)
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "rounds/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert out1.strip() == ""


@pytest.mark.timeout(300)
@pytest.mark.parametrize("n_req", [0, 6])
def test_reference_arm_batched_workload(n_req):
    """The reference arm on a batched workload (4 requests, per-request
    temperatures; --n-req overrides the batch): one line; a step is one full
    request's round and a round of the batch is that many of them."""
    import subprocess

    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "0",
           "--workload", "r4_tiny_mixed"] + (["--n-req", str(n_req)] if n_req else [])
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=280, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    want = n_req or 4
    assert line["impl"] == "reference" and line["config"]["n_req"] == want and line["value"] > 0
    assert f"a round of {want} requests is {want} such rounds" in line["cpu_baseline"]["sample"]
    assert "one full round" in line["cpu_baseline"]["sample"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0
