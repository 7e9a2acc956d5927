"""Multi-replica bookkeeping on the CPU with two gloo ranks: rank discovery,
distinct per-replica request streams, the max-over-replicas time and the
whole-job rate, the reference arm running on rank 0 only, a replica that
dies between steps ending the survivor's next collective with an error, and
one host store shared by the replicas (filled once, mapped by both)."""

import json
import os
import socket
import sys
import time

import pytest

from host_paged_expert_gb300 import replicas

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))


def _timed_worker(rank, world, port, out):
    _env(rank, world, port)
    rep = replicas.from_env()
    replicas.init(rep, "gloo", timeout_s=60)
    replicas.barrier(rep)
    ms = 10.0 + 5.0 * rep.rank  # the last rank is the slow replica
    slow = replicas.max_over_replicas(rep, ms)
    rate = replicas.job_rate(4, rep.world, slow)
    replicas.barrier(rep)
    replicas.finish(rep)
    with open(os.path.join(out, f"r{rank}.json"), "w") as f:
        json.dump({"rank": rep.rank, "root": rep.is_root, "slow": slow, "rate": rate,
                   "seed": replicas.input_seed(0, rep)}, f)


def _dying_worker(rank, world, port, out):
    _env(rank, world, port)
    rep = replicas.from_env()
    replicas.init(rep, "gloo", timeout_s=20)
    replicas.barrier(rep)  # step boundary: both alive
    if rank == 1:
        os._exit(3)  # leaves between steps, nothing in flight
    t0 = time.time()
    try:
        replicas.max_over_replicas(rep, 1.0)
        res = "no error"
    except Exception as e:  # the survivor learns of the loss at its next collective
        res = type(e).__name__
    with open(os.path.join(out, f"r{rank}.json"), "w") as f:
        json.dump({"result": res, "seconds": time.time() - t0}, f)
    os._exit(0)


def _shared_store_worker(rank, world, port, out):
    import numpy as np

    from host_paged_expert_gb300 import shared_store

    _env(rank, world, port)
    rep = replicas.from_env()
    replicas.init(rep, "gloo", timeout_s=60)
    path = os.path.join(out, "store.bin")
    nbytes = 3 * 65536 + 4096
    fills = []

    def fill(store):  # the creator writes every "expert row" once
        fills.append(rank)
        a = np.frombuffer(store.view(), dtype=np.uint8)
        a[:] = (np.arange(nbytes) * 7 % 251).astype(np.uint8)

    store = shared_store.open_for_replicas(rep, path, nbytes, fill)
    a = np.frombuffer(store.view(), dtype=np.uint8)
    same = bool(np.array_equal(a, (np.arange(nbytes) * 7 % 251).astype(np.uint8)))
    aligned = store.ptr % 4096 == 0
    replicas.barrier(rep)
    if rank == 0:  # a write after both mapped it: the other replica sees the same pages, not a copy
        a[12345] = 99
    replicas.barrier(rep)
    seen = int(a[12345])
    replicas.barrier(rep)
    del a
    store.close()
    replicas.barrier(rep)
    replicas.finish(rep)
    with open(os.path.join(out, f"r{rank}.json"), "w") as f:
        json.dump({"filled": fills, "same": same, "aligned": aligned, "seen": seen,
                   "exists": os.path.exists(path)}, f)


def _run(fn, world, tmp_path, limit=120):
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    port = _port()
    ps = [ctx.Process(target=fn, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(limit)
    codes = []
    for p in ps:
        if p.is_alive():
            p.kill()
            p.join()
        codes.append(p.exitcode)
    return codes


def test_from_env_layouts():
    assert replicas.from_env({}) == replicas.Replica(0, 1, 0)
    r = replicas.from_env({"RANK": "3", "WORLD_SIZE": "4", "LOCAL_RANK": "1"})
    assert (r.rank, r.world, r.local_rank, r.is_root) == (3, 4, 1, False)
    for bad in ({"RANK": "2", "WORLD_SIZE": "2"}, {"WORLD_SIZE": "0"}, {"RANK": "-1", "WORLD_SIZE": "2"}):
        with pytest.raises(ValueError):
            replicas.from_env(bad)


def test_job_rate_and_seeds():
    assert replicas.job_rate(8, 1, 1000.0) == pytest.approx(8.0)
    assert replicas.job_rate(8, 4, 500.0) == pytest.approx(64.0)
    with pytest.raises(ValueError):
        replicas.job_rate(1, 1, 0.0)
    seeds = {replicas.input_seed(0, replicas.Replica(r, 8, r)) for r in range(8)}
    assert len(seeds) == 8 and replicas.input_seed(0, replicas.Replica(0, 8, 0)) == 0


def test_two_replicas_gloo(tmp_path):
    pytest.importorskip("torch")
    codes = _run(_timed_worker, 2, tmp_path)
    assert codes == [0, 0]
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert [r["rank"] for r in res] == [0, 1] and [r["root"] for r in res] == [True, False]
    for r in res:  # every rank agrees on the slowest replica's time
        assert r["slow"] == 15.0
        assert r["rate"] == pytest.approx(2 * 4 / 0.015)
    assert res[0]["seed"] == 0 and res[0]["seed"] != res[1]["seed"]


def test_lost_replica_ends_next_collective(tmp_path):
    pytest.importorskip("torch")
    codes = _run(_dying_worker, 2, tmp_path, limit=90)
    assert codes == [0, 3]
    r0 = json.load(open(tmp_path / "r0.json"))
    assert r0["result"] != "no error"
    assert r0["seconds"] < 30


def test_shared_host_store_two_replicas(tmp_path):
    """Replica 0 creates and fills the store; replica 1 maps the filled
    store; both see the same bytes and the same pages; the creator removes
    the file when it closes."""
    pytest.importorskip("torch")
    codes = _run(_shared_store_worker, 2, tmp_path)
    assert codes == [0, 0]
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert res[0]["filled"] == [0] and res[1]["filled"] == []
    assert all(r["same"] and r["aligned"] for r in res)
    assert res[1]["seen"] == 99
    assert not (tmp_path / "store.bin").exists()


def test_reference_arm_only_on_root(capsys):
    sys.path.insert(0, ROOT)
    import bench

    bench.run_reference(None, replicas.Replica(1, 2, 1))  # rank 1: returns without work or output
    assert capsys.readouterr().out == ""
