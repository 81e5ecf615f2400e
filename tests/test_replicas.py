"""The host side of replica runs (one process per GPU, no exchange of data),
exercised with two gloo ranks on the CPU: the launcher's environment, the
barrier, the maximum over ranks of the timed values, and the whole-job rate
(the work of all ranks over the slowest rank's time). bench.py uses these for
`--gpus N` under torchrun."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    from io_aware_exact_tiled_gb300 import replicas
    r, w, loc = replicas.env()
    replicas.init("gloo", w)
    replicas.barrier()
    # each rank reports different times: step time 10 (r + 1) ms and two
    # per-kernel times that disagree in opposite directions
    mx = replicas.max_over_ranks([10.0 * (r + 1), 1.0 + r, 7.0 - r])
    rate = replicas.whole_job_rate(3e12, mx[0] * 1e-3, w)
    assert replicas.active()
    # bench.py's JSON line of a replica run: rank 1 is the slower one
    import contextlib
    import io
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    line = {"value": 100.0 / (r + 1), "ms_per_step": 1.0 * (r + 1), "n_gpus": 1}
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench._emit(line, r, w, "cpu")  # also leaves the process group
    q.put((r, w, loc, mx, rate, True, buf.getvalue()))


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, w, loc, mx, rate, act, printed) in enumerate(out):
        assert (rank, w, loc, act) == (r, world, r, True)
        assert mx == [20.0, 2.0, 7.0]
        # both ranks did 3e12 units; the job took the slower rank's 20 ms
        assert rate == pytest.approx(2 * 3e12 / 0.020)
        if r == 0:
            # 100 units/s at 1 ms per step on rank 0, 2 ms on rank 1: the
            # whole job does 2 x 0.1 units in 2 ms = 100 units/s
            import json
            d = json.loads(printed)
            assert d["n_gpus"] == 2 and d["ms_per_step"] == 2.0
            assert d["value"] == pytest.approx(100.0)
        else:
            assert printed == ""


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    from io_aware_exact_tiled_gb300 import replicas
    assert replicas.env() == (0, 1, 0)
    replicas.init("gloo", 1)  # a single rank joins no process group
    assert not replicas.active()
    assert replicas.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert replicas.whole_job_rate(10.0, 2.0, 1) == 5.0
    with pytest.raises(ValueError):
        replicas.whole_job_rate(1.0, 0.0, 1)
