"""World-size-2 gloo test of bench.py's multi-rank host logic on CPU: the
step time is the max over ranks, the aggregate value counts every rank's
work, and the reference arm prints from rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _body(rank, world, out_q, bench)
    except Exception as e:  # report instead of leaving the parent waiting
        out_q.put((rank, None, None, repr(e)))
    finally:
        dist.destroy_process_group()


def _body(rank, world, out_q, bench):
    if True:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier(ws)
        step_s = 0.010 * (rank + 1)                 # rank 1 is the slow one
        worst = bench.max_over_ranks(step_s, ws)
        flop = 1e12
        value = ws * flop / worst / 1e12            # the aggregate bench.py reports
        buf = io.StringIO()
        with redirect_stdout(buf):
            class A:
                steps, warmup, gpus = 1, 0, world
            bench.reference_arm(A, bench.wl.custom("t", "bf16", 1, 2, 64, 128, 2, 1, seed=1), ws, r)
        out_q.put((rank, worst, value, buf.getvalue()))


def test_two_rank_gloo_host_logic():
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
    (r0, w0, v0, o0), (r1, w1, v1, o1) = res
    assert w0 == w1 == 0.020                       # max over ranks, identical on both
    assert abs(v0 - 2 * 1e12 / 0.020 / 1e12) < 1e-9 and v0 == v1
    assert '"impl": "reference"' in o0 and o1 == ""  # rank 0 alone prints
    import json
    lines = [l for l in o0.splitlines() if l.startswith("{")]
    assert len(lines) == 1                           # one JSON line
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "t"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
