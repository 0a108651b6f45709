"""The expert-parallel exchanges on CPU: two and three gloo ranks.

Each rank routes its own tokens (the oracle's routing of seeded logits), builds
the oracle's dispatch plan, and sends rows carrying (source, assignment,
expert) through the binding's exchange helpers -- the same
torch.distributed all-to-alls the GPU path runs over NCCL.  Checked: the
count exchange, the rows each receiver gets (sources back to back, each
source's segment for it), and that the return exchange delivers every row
back to its sender at its send position.  The device kernels on either side
of the exchanges are covered on the GPU by tests/test_gpu_ep.py.
"""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
E, K = 12, 3


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _tokens(rank):
    return [5, 0, 9][rank]


def _plan(rank, world, shared):
    from oracle import ep as EP
    from oracle import moe as M
    T = _tokens(rank)
    logits = np.random.default_rng(rank).standard_normal((T, E)).astype(np.float32)
    ids, _ = M.route(logits, None, K, True)
    return EP.dispatch_plan(ids, E, world, rank, shared)


def _rank_main(rank, world, port, shared, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import nvfp4_moe_grouped_router_gb300 as nvf
    segs, counts, s2s = _plan(rank, world, shared)
    rows = torch.tensor([[rank, a, e] for r in range(world) for a, e in segs[r]], dtype=torch.int64).reshape(-1, 3)
    send_counts = torch.from_numpy(counts.astype(np.int32))
    recv_counts = nvf.ep_exchange_counts(send_counts)
    send_splits = send_counts.sum(dim=1).tolist()
    recv_splits = recv_counts.sum(dim=1).tolist()
    recv = nvf.ep_exchange_rows(rows, send_splits, recv_splits)
    # the receiver "computes": its result row for an arrival is the arrival itself
    back = nvf.ep_exchange_rows(recv, recv_splits, send_splits)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"recv_counts": recv_counts.tolist(), "recv": recv.tolist(), "back": back.tolist(),
                   "s2s": s2s.tolist()}, f)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,shared", [(2, False), (2, True), (3, True)])
def test_exchange_round_trip(tmp_path, world, shared):
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, shared, str(tmp_path)), nprocs=world, start_method="spawn")
    sys.path.insert(0, ROOT)
    plans = [_plan(r, world, shared) for r in range(world)]
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in range(world):
        # receiver r got source s's count row for r, and source s's segment for r, sources in order
        assert res[r]["recv_counts"] == [plans[s][1][r].tolist() for s in range(world)]
        expect = [[s, a, e] for s in range(world) for a, e in plans[s][0][r]]
        assert res[r]["recv"] == expect
    for s in range(world):
        # every row came back to its sender, at its send position
        back = np.array(res[s]["back"], dtype=np.int64).reshape(-1, 3)
        s2s = np.array(res[s]["s2s"])
        for a, pos in enumerate(s2s):
            assert back[pos, 0] == s and back[pos, 1] == a


def test_local_scales():
    sys.path.insert(0, ROOT)
    import nvfp4_moe_grouped_router_gb300 as nvf
    gs = torch.arange(13, dtype=torch.float32)
    assert nvf.ep_local_scales(gs, 12, 4, 2, True).tolist() == [6.0, 7.0, 8.0, 12.0]
    assert nvf.ep_local_scales(gs[:12], 12, 3, 0, False).tolist() == [0.0, 1.0, 2.0, 3.0]
