"""The N > 1 plumbing on CPU: world_size-2 gloo process groups.

The data path has no collective; these check the sharding and the
measurement collectives (barrier, max / sum over ranks) that bench.py uses
when it runs one process per GPU, and that a rank's share decodes the same
rows as the single-process run (oracle decoder on CPU, sharded ids)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from lossless_invariant_bit_gb300 import dist as ibpdist


def test_shard_tiles_range():
    for n in [0, 1, 7, 200_000, 200_001]:
        for world in [1, 2, 3, 8]:
            got = [ibpdist.shard(n, r, world) for r in range(world)]
            assert sum(c for _, c in got) == n
            pos = 0
            for s, c in got:
                assert s == pos
                pos += c
            counts = [c for _, c in got]
            assert max(counts) - min(counts) <= 1
    with pytest.raises(ValueError):
        ibpdist.shard(10, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = ibpdist.rank_world()
        assert (r, lr, w) == (rank, rank, world)
        dist.barrier()
        mx = ibpdist.max_over_ranks(1.5 + rank, dist)
        sm = ibpdist.sum_over_ranks(10.0 * (rank + 1), dist)
        # a rank's share of a batch, decoded by the oracle on the CPU
        from lossless_invariant_bit_gb300 import workloads as wl
        from oracle import ref_c
        n_rows, R, C = 3000, 512, 1024
        rows = wl.sparse_gnn_rows(n_rows, seed=4)
        rb = rows.view(np.uint8)
        m, b = ref_c.build_meta(rb, 95, 100)
        slots = np.zeros((n_rows, R), np.uint8)
        bm = np.zeros((n_rows + 31) // 32, np.uint32)
        ref_c.compress_batch(rb, C, m, b, slots, bm)
        ids = wl.uniform_ids(1001, n_rows, seed=0)
        s, c = ibpdist.shard(len(ids), rank, world)
        out, bad = ref_c.decompress_batch(slots, bm, R, C, m, b, ids=ids[s:s + c], slot_stride=R)
        ok = bad == 0 and np.array_equal(out, rb[ids[s:s + c]])
        q.put((rank, mx, sm, c, ok))
    finally:
        dist.destroy_process_group()


def test_gloo_world2_measurement_collectives():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]
    assert [r[2] for r in res] == [30.0, 30.0]
    assert sum(r[3] for r in res) == 1001
    assert all(r[4] for r in res)
