"""Multi-rank host logic on CPU (gloo, world size 2): the step time is the
max over ranks and only rank 0 reports (bench.py); a problem's heads split
over the ranks with vsa_head_slice cover every head exactly once with each
GQA group inside one rank. Ranks are spawned as separate processes."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    m = bench.reduce_max(10.0 + rank * 5.0, ws, torch.device("cpu"))
    out.put((rank, m))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}


def test_reference_arm_other_ranks_print_nothing(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        gpus, steps, warmup = 2, 1, 3
    bench.reference_arm(A())
    assert capsys.readouterr().out == ""


def test_single_rank_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1, None) == 3.5


def _slice_worker(rank, world, port, hq, hkv, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from bwd_tile_mean_gb300 import vsa
    d = vsa.VsaDesc(1, 0, 1, hq, hkv, 128, 76800, 76800, 256, 256, 300, 300, None, None, 0.0)
    s, q0, kv0 = vsa.vsa_head_slice(d, world, rank)
    mine = torch.tensor([q0, s.Hq, kv0, s.Hkv], dtype=torch.int64)
    every = [torch.zeros(4, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(every, mine)
    out.put((rank, [x.tolist() for x in every]))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("hq,hkv", [(40, 40), (12, 2)])
def test_head_slices_cover_every_head_once_over_two_gloo_ranks(hq, hkv):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_slice_worker, args=(r, 2, port, hq, hkv, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res[0] == res[1]                       # every rank sees the same split
    g = hq // hkv
    qheads, kvheads = [], []
    for q0, nq, kv0, nkv in res[0]:
        qheads += range(q0, q0 + nq)
        kvheads += range(kv0, kv0 + nkv)
        assert nq == nkv * g and q0 == kv0 * g    # whole GQA groups: query head h reads KV head h // g
    assert sorted(qheads) == list(range(hq)) and sorted(kvheads) == list(range(hkv))
