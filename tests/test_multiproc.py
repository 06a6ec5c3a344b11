"""Two ranks on CPU (gloo): each rank builds its own trees through the C ABI
(metadata-only pools), checks its allocator state against the oracle, and the
ranks combine their step times by max and their branch counts by sum -- the
host-side logic of a multi-GPU run, with no collective on the data path."""

import multiprocessing as mp
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import torch.distributed as dist

    from oracle import replay as rp
    from paged_kv_cache_attn_gb300 import harness as H
    from paged_kv_cache_attn_gb300 import workloads as W

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = W.make("deep_tree", rank, root_tokens=200, depth=3, min_seg=5,
                   max_seg=40)
        lib = H.Cache(w, with_data=False)
        ref = rp.replay(w, with_data=False)
        same = (lib.refcounts() == ref.model.ref and
                lib.free_stack() == ref.model.free_stack() and
                lib.decode_ids == ref.decode_ids and
                lib.evicted == ref.evicted)
        t = torch.tensor([1.5 + rank])             # this rank's step time
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        n = torch.tensor([len(lib.decode_ids)])
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
        seeds = [None] * world
        dist.all_gather_object(seeds, w.seed)
        out.put((rank, same, float(t.item()), int(n.item()), seeds,
                 len(lib.decode_ids)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(r[1] for r in res)                 # state matches the oracle
    assert all(r[2] == 2.5 for r in res)          # max over ranks
    assert res[0][3] == res[0][5] + res[1][5]     # branches summed
    assert res[0][4][0] != res[0][4][1]           # distinct trees per rank
