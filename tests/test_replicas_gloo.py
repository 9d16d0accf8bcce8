"""The bench's N > 1 path on the host: independent replicas (one per rank), timed steps
reduced to the slowest rank, and the job's rate counted over every rank's tokens.  Two gloo
ranks on CPU (the decode path has no exchange step, so no collective touches the data)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from routed_expert_ffn_gemv_gb300 import synth
        cfg = synth.config(1)
        ms = 100.0 + 50.0 * rank  # rank 1 is the slower replica
        ms_max = bench.max_over_ranks(ms, world, torch)
        st = {"queries": [10 * 8], "hits": [0], "h2d_bytes": 8 * 10 * cfg.expert_bytes,
              "route_hits": 0, "route_queries": 8 * 8 * 10}
        peaks = {"hbm_gbs": 6784.5}
        r = bench.batch_result(cfg, 8, 10, ms_max, st, world, peaks, 211.0)
        out.put((rank, ms_max, r["tokens_per_s"], r["frac_of_measured_hbm_roofline"]))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_count_every_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    # both ranks see the slowest rank's time
    assert [r[1] for r in res] == [150.0, 150.0]
    # whole-job rate: 2 replicas x 8 tokens x 10 steps in 150 ms
    assert res[0][2] == pytest.approx(2 * 8 * 10 / 0.150)
    assert res[0][2] == res[1][2]
    # the per-GPU fraction of the roofline does not grow with the replica count
    r1 = res[0][3]
    assert 0 < r1 < 1
