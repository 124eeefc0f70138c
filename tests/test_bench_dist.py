"""The multi-rank bookkeeping of bench.py on CPU: two gloo ranks agree on the
max-over-ranks step time and the summed cache bytes, and every rank decodes its own
batch (same shape, its own seed), as the weak-scaling contract requires."""

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W

    d = bench.Dist(backend="gloo")
    w = bench.rank_workload(W.WORKLOADS["v2_b32_l4096"], d.rank)
    step_ms = 1.0 + d.rank                          # rank 1 is the slow one
    cache_bytes = W.cache_bytes(w)
    d.barrier()
    mx = d.max(step_ms)
    total = d.sum(cache_bytes)
    q0 = W.gen_q(w)[0, 0, :4].tolist()
    d.close()
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(repr((mx, total, w.seed, w.batch, w.ctx, q0)))


def test_two_gloo_ranks(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    r0 = eval((tmp_path / "r0.txt").read_text())
    r1 = eval((tmp_path / "r1.txt").read_text())
    assert r0[0] == r1[0] == 2.0                     # max over ranks
    assert r0[1] == r1[1] == 2 * 32 * 4096 * 1152    # both ranks' cache bytes
    assert r0[2] != r1[2]                            # own seed per rank
    assert r0[3:5] == r1[3:5] == (32, 4096)          # same shape
    assert r0[5] != r1[5]                            # hence different inputs
