"""The multi-replica timing of bench.py on CPU: two gloo ranks, max over ranks, whole-job value."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    secs = [0.5, 0.75][rank]
    worst = bench.max_over_ranks(secs, "cpu")
    dist.barrier()
    q.put((rank, worst, bench.whole_job_gbs(10 ** 9, world, worst / 10)))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, worst, gbs in got:
        assert worst == 0.75                       # both ranks see the slowest rank's time
        assert gbs == pytest.approx(2 * 1e9 / 0.075 / 1e9)   # two replicas' bytes over that time


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod_hash", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    return bench


def test_profile_hash_ignores_comments_not_code():
    """A profile's traffic stays valid across documentation edits of the kernel
    source, and goes stale when the code itself changes."""
    bench = _bench_module()
    src = b"__device__ int f(int a) {\n  return a + 1;  // one more\n}\n"
    doc = b"// what f does\n__device__ int f(int a) {\n  /* unchanged */ return a + 1;\n}\n"
    code = b"__device__ int f(int a) {\n  return a + 2;\n}\n"
    assert bench._code_only(src) == bench._code_only(doc)
    assert bench._code_only(src) != bench._code_only(code)
