"""Multi-process slicing on CPU ranks (gloo, world size 2; no GPU).

Slices are independent sub-contractions whose results add up ("Crossing
the single-GPU memory wall", section 1.1), so R processes can each take the
slices shard_slices assigns them and sum their outputs once.  Here every
rank contracts its shard with the fp64 oracle, the ranks all-reduce the
partial results over gloo, and rank 0 compares with the unsliced oracle
value.  This tests the partition and the reduction the GPU ranks use.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import exact_tensor_network_gb300 as tn


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import oracle
    from workloads import choose_slices, greedy_tree, largest_intermediate, random_network
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        net = random_network(30, 4)
        tree = greedy_tree(net, 0)
        sl = choose_slices(net, tree, largest_intermediate(net, tree) // 8)[:3]
        ext = [net.extents[x] for x in sl]
        n_slices = int(np.prod(ext))
        first, step, count = tn.shard_slices(n_slices, rank, world)
        part = np.zeros([net.extents[x] for x in net.open_modes], dtype=np.complex128)
        for sigma in range(first, n_slices, step):
            vals = np.unravel_index(sigma, ext)
            t2, d2 = oracle.slice_leaves(net.tensors, net.data, sl, [int(v) for v in vals])
            part = part + oracle.contract(t2, net.extents, net.open_modes, d2, tree)
        buf = torch.from_numpy(np.stack([part.real, part.imag]).copy())
        dist.all_reduce(buf, op=dist.ReduceOp.SUM)
        if rank == 0:
            total = buf[0].numpy() + 1j * buf[1].numpy()
            full = oracle.contract(net.tensors, net.extents, net.open_modes, net.data, tree)
            err = float(np.abs(total - full).max() / np.abs(full).max())
            q.put((n_slices, err))
    finally:
        dist.destroy_process_group()


def test_shard_slices_partition():
    for n in (1, 2, 7, 8, 64):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                first, step, count = tn.shard_slices(n, r, world)
                mine = list(range(first, n, step))
                assert len(mine) == count
                seen += mine
            assert sorted(seen) == list(range(n))
    with pytest.raises(ValueError):
        tn.shard_slices(4, 2, 2)


def test_two_gloo_ranks_sum_their_slices():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    n_slices, err = q.get(timeout=10)
    assert n_slices >= 2
    assert err <= 1e-12
