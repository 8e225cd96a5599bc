"""Fused multi-store gather (ibp_group_*) against the rows and the per-store path.

A DLRM-shaped group (26 tables, Zipf lookups, [batch, tables, dim] output)
and a mixed group whose stores cover every decode mode (uniform, two-run,
network, all-raw), host and HBM sources, raw chunks and an out-of-range id.
"""
import numpy as np
import pytest
import torch

from lossless_invariant_bit_gb300 import ibp
from lossless_invariant_bit_gb300 import workloads as wl
from oracle import ref_c
from tests.gpu_util import DEV, Store, oracle_slots, rows_u8, to_dev

pytestmark = pytest.mark.gpu


def _host_store(R, C, rows_b, sample=None, num=95, den=100, host=True):
    n = rows_b.shape[0]
    st = Store(R, C, n)
    d = torch.from_numpy(rows_b).to(DEV)
    ids = None if sample is None else torch.from_numpy(sample).to(DEV)
    ibp.ibp_build_meta(st.h, d, R, ids, n if sample is None else len(sample), num, den)
    slots = (torch.empty((n, st.slot), dtype=torch.uint8, pin_memory=True) if host
             else torch.empty((n, st.slot), dtype=torch.uint8, device=DEV))
    ibp.ibp_compress(st.h, slots, d, R, None, n, None)
    torch.cuda.synchronize()
    return st, slots


@pytest.mark.parametrize("dim", [128, 512])
def test_group_dlrm_matches_per_store(dim):
    T, N, B, R, C = 26, 5000, 2049, dim * 4, 1024
    stores, slots, tables = [], [], []
    try:
        for t in range(T):
            rb = rows_u8(wl.dlrm_rows(N, dim, table=t, seed=1))
            st, sl = _host_store(R, C, rb, wl.sample_ids(N, 50, seed=t), host=(t % 3 != 0))
            stores.append(st)
            slots.append(sl)
            tables.append(rb)
        ids = np.stack([wl.zipf_ids(B, N, table=t, seed=2) for t in range(T)], axis=1)
        grp = ibp.ibp_group_create([s.h for s in stores], slots)
        try:
            out = torch.full((B, T, R), 0xCC, dtype=torch.uint8, device=DEV)
            ibp.ibp_group_gather_decompress(grp, out, T * R, to_dev(ids), B)
            for s in stores:
                assert s.status() == ibp.IBP_OK
            o = out.cpu().numpy()
            for t in range(T):
                assert np.array_equal(o[:, t], tables[t][ids[:, t]]), t
            # the per-store strided gathers give the same bytes
            ref = torch.zeros((B, T, R), dtype=torch.uint8, device=DEV)
            for t in range(T):
                ibp.ibp_gather_decompress_strided(stores[t].h, ref[:, t], T * R, slots[t], None,
                                                  to_dev(np.ascontiguousarray(ids[:, t])), B)
            assert torch.equal(out, ref)
        finally:
            ibp.ibp_group_destroy(grp)
    finally:
        for s in stores:
            s.close()


def test_group_mixed_modes_errors_and_raw_chunks():
    R, C, N, B = 512, 64, 3000, 777
    stores, slots, tables = [], [], []
    specs = []
    try:
        # uniform two-run (dense fp32), uniform with empty ~Mask (sparse), network (fuzz),
        # two-run non-uniform (set), all raw (fresh store), uniform one run (1 + k/1024)
        dense = rows_u8(wl.dense_gnn_rows(N, seed=3))
        sparse = rows_u8(wl.sparse_gnn_rows(N, seed=3))
        fuzz = wl.fuzz_rows(N, R, seed=4)
        tiny = rows_u8(wl.tiny_rows(seed=5, n_rows=N, dim=R // 4, raw_frac=0.02)[0])
        for rb, host in [(dense, True), (sparse, False), (fuzz, True), (tiny, False)]:
            st, sl = _host_store(R, C, rb, host=host)
            stores.append(st)
            slots.append(sl)
            tables.append(rb)
        # two-run, non-uniform Masks, set on the host; a tenth of the rows miss one word
        g = np.random.default_rng(6)
        mask = np.zeros(R // 4, np.uint32)
        for w in range(R // 4):
            a0 = int(g.integers(0, 16))
            keep = ((1 << int(g.integers(1, 9))) - 1) << a0 | (1 << 31)
            mask[w] = ~np.uint32(keep & 0xFFFFFFFF)
        bitval = g.integers(0, 1 << 32, size=R // 4, dtype=np.uint64).astype(np.uint32) & mask
        rows = (g.integers(0, 1 << 32, size=(N, R // 4), dtype=np.uint64).astype(np.uint32)
                & ~mask) | bitval
        miss = g.random(N) < 0.1
        rows[miss, 3] ^= mask[3] & 0x00FF0000
        rb = rows.view(np.uint8)
        st = Store(R, C, N)
        st.set_meta(mask, bitval)
        assert ibp.ibp_store_get_info(st.h).max_runs <= 2
        sl = torch.empty((N, st.slot), dtype=torch.uint8, pin_memory=True)
        ibp.ibp_compress(st.h, sl, torch.from_numpy(rb).to(DEV), R, None, N, None)
        stores.append(st)
        slots.append(sl)
        tables.append(rb)
        # all raw: a store whose Mask was never built
        st = Store(R, C, N)
        sl = torch.empty((N, st.slot), dtype=torch.uint8, device=DEV)
        ibp.ibp_compress(st.h, sl, torch.from_numpy(fuzz).to(DEV), R, None, N, None)
        stores.append(st)
        slots.append(sl)
        tables.append(fuzz)
        torch.cuda.synchronize()
        T = len(stores)
        ids = np.stack([g.integers(0, N, size=B) for _ in range(T)], axis=1).astype(np.int64)
        ids[5, 2] = N + 7  # out of range in store 2
        grp = ibp.ibp_group_create([s.h for s in stores], slots)
        try:
            stride = T * R + 64
            out = torch.full((B, stride), 0xCC, dtype=torch.uint8, device=DEV)
            ibp.ibp_group_gather_decompress(grp, out, stride, to_dev(ids), B)
            st_codes = [s.status() for s in stores]
            assert st_codes[2] == ibp.IBP_ERANGE
            assert all(c == ibp.IBP_OK for i, c in enumerate(st_codes) if i != 2)
            o = out.cpu().numpy()
            for t in range(T):
                got = o[:, t * R:(t + 1) * R]
                want = tables[t][np.clip(ids[:, t], 0, N - 1)]
                if t == 2:
                    assert np.all(got[5] == 0)
                    got = np.delete(got, 5, axis=0)
                    want = np.delete(want, 5, axis=0)
                assert np.array_equal(got, want), t
            assert np.all(o[:, T * R:] == 0xCC)  # bytes past the last table untouched
        finally:
            ibp.ibp_group_destroy(grp)
    finally:
        for s in stores:
            s.close()


def test_group_rejects_mixed_geometry():
    a = Store(512, 256, 10)
    b = Store(1024, 256, 10)
    c = Store(4096, 256, 10)
    try:
        buf = torch.empty(10 * 4096, dtype=torch.uint8, device=DEV)
        with pytest.raises(ibp.IbpError) as e:
            ibp.ibp_group_create([a.h, b.h], [buf, buf])
        assert e.value.status == ibp.IBP_EINVAL
        with pytest.raises(ibp.IbpError) as e:  # rows above 2 KB are not fused
            ibp.ibp_group_create([c.h], [buf])
        assert e.value.status == ibp.IBP_EINVAL
    finally:
        for s in (a, b, c):
            s.close()


def test_group_ordered_matches_group():
    """The ordered group gather (items bucketed by store and region) writes the
    plain group gather's bytes and status codes, an out-of-range id included."""
    R, C, N, B = 512, 1024, 4000, 1500
    stores, slots, tables = [], [], []
    try:
        for t in range(5):
            rb = rows_u8(wl.dlrm_rows(N, R // 4, table=t, seed=7))
            st, sl = _host_store(R, C, rb, wl.sample_ids(N, 50, seed=t), host=(t != 2))
            stores.append(st)
            slots.append(sl)
            tables.append(rb)
        T = len(stores)
        ids = np.stack([wl.zipf_ids(B, N, table=t, seed=8) for t in range(T)], axis=1)
        ids[7, 3] = -4  # out of range in store 3
        grp = ibp.ibp_group_create([s.h for s in stores], slots)
        try:
            stride = T * R + 32
            ref = torch.full((B, stride), 0x33, dtype=torch.uint8, device=DEV)
            ibp.ibp_group_gather_decompress(grp, ref, stride, to_dev(ids), B)
            codes = [s.status() for s in stores]
            assert codes[3] == ibp.IBP_ERANGE
            out = torch.full((B, stride), 0x33, dtype=torch.uint8, device=DEV)
            ws = torch.empty(ibp.order_workspace_bytes(B * T), dtype=torch.uint8, device=DEV)
            ibp.ibp_group_gather_decompress_ordered(grp, out, stride, to_dev(ids), B, ws,
                                                    ws.numel())
            assert [s.status() for s in stores] == codes
            assert torch.equal(out, ref)
            o = out.cpu().numpy()
            for t in range(T):
                ok = ids[:, t] >= 0
                assert np.array_equal(o[ok, t * R:(t + 1) * R], tables[t][ids[ok, t]]), t
            with pytest.raises(ibp.IbpError) as e:
                ibp.ibp_group_gather_decompress_ordered(grp, out, stride, to_dev(ids), B, ws,
                                                        ws.numel() - 16)
            assert e.value.status == ibp.IBP_EINVAL
        finally:
            ibp.ibp_group_destroy(grp)
    finally:
        for s in stores:
            s.close()


def test_group_length_tables_and_a_rebuilt_store():
    """2 KB rows at 1 KB chunks: about half the rows carry one raw chunk, so
    their streams are longer than the shortest one.  With each store's length
    table attached before the group is made, the first fetch takes the whole
    stream; the output is the same.  A store whose Mask/Bitval is rebuilt
    after the group was made reports IBP_EINVAL and its lookups are
    zero-filled; the other stores are unaffected."""
    T, N, B, dim, C = 5, 4000, 1500, 512, 1024
    R = dim * 4
    stores, slots, tables, lengths = [], [], [], []
    try:
        for t in range(T):
            rb = rows_u8(wl.dlrm_rows(N, dim, table=t, seed=7))
            st = Store(R, C, N)
            d = torch.from_numpy(rb).to(DEV)
            smp = torch.from_numpy(wl.sample_ids(N, 100, seed=t)).to(DEV)
            ibp.ibp_build_meta(st.h, d, R, smp, smp.numel(), 95, 100)
            sl = torch.empty((N, st.slot), dtype=torch.uint8, pin_memory=True)
            ln = torch.empty(N, dtype=torch.int32, device=DEV)
            ibp.ibp_compress(st.h, sl, d, R, None, N, ln)
            torch.cuda.synchronize()
            ibp.ibp_store_set_lengths(st.h, ln)
            stores.append(st)
            slots.append(sl)
            tables.append(rb)
            lengths.append(ln)
        ln_np = lengths[0].cpu().numpy()
        min_bytes = int(ln_np[ln_np < R].min())
        assert (ln_np[ln_np < R] > min_bytes).mean() > 0.2  # many rows need more than the shortest stream
        ids = np.stack([wl.zipf_ids(B, N, table=t, seed=3) for t in range(T)], axis=1)
        grp = ibp.ibp_group_create([s.h for s in stores], slots)
        try:
            out = torch.full((B, T, R), 0xCC, dtype=torch.uint8, device=DEV)
            ibp.ibp_group_gather_decompress(grp, out, T * R, to_dev(ids), B)
            for s in stores:
                assert s.status() == ibp.IBP_OK
            o = out.cpu().numpy()
            for t in range(T):
                assert np.array_equal(o[:, t], tables[t][ids[:, t]]), t
            ws = torch.empty(ibp.order_workspace_bytes(B * T), dtype=torch.uint8, device=DEV)
            out2 = torch.zeros_like(out)
            ibp.ibp_group_gather_decompress_ordered(grp, out2, T * R, to_dev(ids), B, ws,
                                                    ws.numel())
            assert torch.equal(out, out2)
            # store 2 gets a new Mask/Bitval: the group's copy of its properties is stale
            d2 = torch.from_numpy(tables[2]).to(DEV)
            ibp.ibp_build_meta(stores[2].h, d2, R, None, N, 1, 1)
            torch.cuda.synchronize()
            out.fill_(0xCC)
            ibp.ibp_group_gather_decompress(grp, out, T * R, to_dev(ids), B)
            assert stores[2].status() == ibp.IBP_EINVAL
            for t in (0, 1, 3, 4):
                assert stores[t].status() == ibp.IBP_OK
            o = out.cpu().numpy()
            assert not o[:, 2].any()
            for t in (0, 1, 3, 4):
                assert np.array_equal(o[:, t], tables[t][ids[:, t]]), t
        finally:
            ibp.ibp_group_destroy(grp)
    finally:
        for s in stores:
            s.close()


def test_group_ordered_repeats_large_buckets_and_errors():
    """The ordered group gather over heavy repeats: every item equals the plain
    group gather's (bytes and status codes) and the rows.  Store 0 (dense,
    uniform, host) has one row whose stream is corrupt, looked up 2600 times:
    its bucket is above the 2048 items grouped in shared memory and stays in
    scatter order, and the repeats of a corrupt row are zero-filled like the
    row.  Store 1 (network mode, host) has a hot row whose repeats span warp
    shares; store 2 (two-run mode, HBM) has out-of-range ids repeated next to
    each other; store 3 (all raw, HBM) takes the raw path with repeats.  A
    batch of 3 leaves most warps an empty share."""
    R, C, N, B = 512, 64, 3000, 6000
    g = np.random.default_rng(11)
    stores, slots, tables = [], [], []
    try:
        dense = rows_u8(wl.dense_gnn_rows(N, seed=13))
        fuzz = wl.fuzz_rows(N, R, seed=14)
        tiny = rows_u8(wl.tiny_rows(seed=15, n_rows=N, dim=R // 4, raw_frac=0.02)[0])
        for rb, host in [(dense, True), (fuzz, True), (tiny, False)]:
            st, sl = _host_store(R, C, rb, host=host)
            stores.append(st)
            slots.append(sl)
            tables.append(rb)
        st = Store(R, C, N)  # all raw: a store whose Mask was never built
        sl = torch.empty((N, st.slot), dtype=torch.uint8, device=DEV)
        ibp.ibp_compress(st.h, sl, torch.from_numpy(fuzz).to(DEV), R, None, N, None)
        stores.append(st)
        slots.append(sl)
        tables.append(fuzz)
        torch.cuda.synchronize()
        # a packed row of store 0 made corrupt: every chunk flagged raw in its header
        bm = stores[0].bitmap()
        packed = [i for i in range(N) if not (int(bm[i >> 5]) >> (i & 31)) & 1]
        bad = packed[len(packed) // 2]
        slots[0][bad, :4] = 0
        T = len(stores)
        ids = np.stack([wl.zipf_ids(B, N, table=t, seed=16) for t in range(T)], axis=1)
        ids[g.choice(B, 2600, replace=False), 0] = bad
        ids[g.choice(B, 900, replace=False), 1] = int(ids[0, 1])
        ids[100:140, 2] = N + 5
        ids[200:230, 2] = -1
        grp = ibp.ibp_group_create([s.h for s in stores], slots)
        try:
            for b in (B, 3):
                sub = np.ascontiguousarray(ids[:b])
                ref = torch.full((b, T, R), 0xCC, dtype=torch.uint8, device=DEV)
                ibp.ibp_group_gather_decompress(grp, ref, T * R, to_dev(sub), b)
                codes = [s.status() for s in stores]
                out = torch.full((b, T, R), 0x33, dtype=torch.uint8, device=DEV)
                ws = torch.empty(ibp.order_workspace_bytes(b * T), dtype=torch.uint8,
                                 device=DEV)
                ibp.ibp_group_gather_decompress_ordered(grp, out, T * R, to_dev(sub), b, ws,
                                                        ws.numel())
                assert [s.status() for s in stores] == codes, b
                assert torch.equal(out, ref), b
                o = out.cpu().numpy()
                for t in range(T):
                    x = sub[:, t]
                    ok = (x >= 0) & (x < N) & ~((t == 0) & (x == bad))
                    assert np.array_equal(o[ok, t], tables[t][x[ok]]), (b, t)
                    assert not o[~ok, t].any(), (b, t)
                if b == B:
                    assert codes[0] == ibp.IBP_ECORRUPT and codes[2] == ibp.IBP_ERANGE
                    assert codes[1] == ibp.IBP_OK and codes[3] == ibp.IBP_OK
        finally:
            ibp.ibp_group_destroy(grp)
    finally:
        for s in stores:
            s.close()


def test_group_planned_gathers():
    """A plan made ahead (ibp_group_order_plan) and its gather
    (ibp_group_gather_decompress_planned) write the plain group gather's
    bytes and status codes, an out-of-range id included:
    - on one stream;
    - three batches pipelined over two streams and two workspaces, each
      batch's plan made while the previous batch is gathered;
    - with a plan made for other ids of the same size (the rows are right);
    - a workspace holding no plan, or a plan for another batch size: the
      gather writes nothing and store 0 reports IBP_EINVAL."""
    R, C, N, B = 512, 1024, 4000, 1500
    stores, slots, tables = [], [], []
    try:
        for t in range(5):
            rb = rows_u8(wl.dlrm_rows(N, R // 4, table=t, seed=61))
            st, sl = _host_store(R, C, rb, wl.sample_ids(N, 50, seed=t), host=(t != 2))
            stores.append(st)
            slots.append(sl)
            tables.append(rb)
        T = len(stores)
        batches = []
        for k in range(3):
            ids = np.stack([wl.zipf_ids(B, N, table=t, seed=62 + k) for t in range(T)], axis=1)
            batches.append(ids)
        batches[1][9, 3] = N + 2  # out of range in store 3
        grp = ibp.ibp_group_create([s.h for s in stores], slots)
        try:
            wsb = ibp.order_workspace_bytes(B * T)
            ws = [torch.zeros(wsb, dtype=torch.uint8, device=DEV) for _ in range(2)]
            dev_ids = [to_dev(x) for x in batches]
            refs, codes = [], []
            for x in dev_ids:
                ref = torch.full((B, T, R), 0xCC, dtype=torch.uint8, device=DEV)
                ibp.ibp_group_gather_decompress(grp, ref, T * R, x, B)
                refs.append(ref)
                codes.append([s.status() for s in stores])
            assert codes[1][3] == ibp.IBP_ERANGE and codes[0] == [ibp.IBP_OK] * T
            # one stream
            out = torch.full((B, T, R), 0x33, dtype=torch.uint8, device=DEV)
            ibp.ibp_group_order_plan(grp, dev_ids[1], B, ws[0], wsb)
            ibp.ibp_group_gather_decompress_planned(grp, out, T * R, dev_ids[1], B, ws[0], wsb)
            assert [s.status() for s in stores] == codes[1]
            assert torch.equal(out, refs[1])
            # pipelined: batch k+1 planned on a second stream while batch k is gathered
            gs, ps = torch.cuda.Stream(), torch.cuda.Stream()
            outs = [torch.full((B, T, R), 0x33, dtype=torch.uint8, device=DEV) for _ in range(3)]
            planned = [torch.cuda.Event() for _ in range(3)]
            gathered = [torch.cuda.Event() for _ in range(3)]
            gs.wait_stream(torch.cuda.current_stream())
            ps.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(ps):
                ibp.ibp_group_order_plan(grp, dev_ids[0], B, ws[0], wsb, ps)
                planned[0].record(ps)
            for k in range(3):
                with torch.cuda.stream(gs):
                    gs.wait_event(planned[k])
                    ibp.ibp_group_gather_decompress_planned(grp, outs[k], T * R, dev_ids[k], B,
                                                            ws[k % 2], wsb, gs)
                    gathered[k].record(gs)
                if k + 1 < 3:
                    with torch.cuda.stream(ps):
                        if k >= 1:
                            ps.wait_event(gathered[k - 1])  # its workspace is free again
                        ibp.ibp_group_order_plan(grp, dev_ids[k + 1], B, ws[(k + 1) % 2], wsb, ps)
                        planned[k + 1].record(ps)
            torch.cuda.synchronize()
            for k in range(3):
                assert torch.equal(outs[k], refs[k]), k
            assert [s.status() for s in stores] == [max(c) for c in zip(*codes)]
            # a plan for batch 0's ids, gathered with batch 2's: right rows
            ibp.ibp_group_order_plan(grp, dev_ids[0], B, ws[0], wsb)
            out.fill_(0x33)
            ibp.ibp_group_gather_decompress_planned(grp, out, T * R, dev_ids[2], B, ws[0], wsb)
            assert [s.status() for s in stores] == [ibp.IBP_OK] * T
            assert torch.equal(out, refs[2])
            o = out.cpu().numpy()
            for t in range(T):
                assert np.array_equal(o[:, t], tables[t][batches[2][:, t]]), t
            # no plan in the workspace, or one for another batch size
            fresh = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
            other = torch.zeros(ibp.order_workspace_bytes(B * T), dtype=torch.uint8, device=DEV)
            ibp.ibp_group_order_plan(grp, dev_ids[0][:B - 100].contiguous(), B - 100, other,
                                     other.numel())
            for w in (fresh, other):
                out.fill_(0x33)
                ibp.ibp_group_gather_decompress_planned(grp, out, T * R, dev_ids[2], B, w, wsb)
                assert stores[0].status() == ibp.IBP_EINVAL
                assert [s.status() for s in stores[1:]] == [ibp.IBP_OK] * (T - 1)
                assert bool((out == 0x33).all())
            with pytest.raises(ibp.IbpError) as e:
                ibp.ibp_group_gather_decompress_planned(grp, out, T * R, dev_ids[2], B, ws[0],
                                                        wsb - 16)
            assert e.value.status == ibp.IBP_EINVAL
        finally:
            ibp.ibp_group_destroy(grp)
    finally:
        for s in stores:
            s.close()


@pytest.mark.parametrize("B", [16384, 20000])
def test_group_ordered_large_batches(B):
    """Batches of 16384 and 20000 rows over two stores (one in host memory,
    one in HBM): Zipf lookups with a row repeated 3000 times, whose bucket
    holds more items than are grouped in shared memory; the plain group
    gather's bytes and the rows."""
    R, C, N, T = 512, 1024, 6000, 2
    stores, slots, tables = [], [], []
    try:
        for t in range(T):
            rb = rows_u8(wl.dlrm_rows(N, R // 4, table=t, seed=51))
            st, sl = _host_store(R, C, rb, host=(t == 0))
            stores.append(st)
            slots.append(sl)
            tables.append(rb)
        ids = np.stack([wl.zipf_ids(B, N, table=t, seed=52) for t in range(T)], axis=1)
        ids[np.random.default_rng(53).choice(B, 3000, replace=False), 1] = 17
        grp = ibp.ibp_group_create([s.h for s in stores], slots)
        try:
            ref = torch.full((B, T, R), 0xCC, dtype=torch.uint8, device=DEV)
            ibp.ibp_group_gather_decompress(grp, ref, T * R, to_dev(ids), B)
            out = torch.full((B, T, R), 0x33, dtype=torch.uint8, device=DEV)
            ws = torch.empty(ibp.order_workspace_bytes(B * T), dtype=torch.uint8, device=DEV)
            ibp.ibp_group_gather_decompress_ordered(grp, out, T * R, to_dev(ids), B, ws,
                                                    ws.numel())
            for s in stores:
                assert s.status() == ibp.IBP_OK
            assert torch.equal(out, ref)
            o = out.cpu().numpy()
            for t in range(T):
                assert np.array_equal(o[:, t], tables[t][ids[:, t]]), t
        finally:
            ibp.ibp_group_destroy(grp)
    finally:
        for s in stores:
            s.close()


@pytest.mark.parametrize("T", [1, 64])
def test_group_ordered_one_and_most_tables(T):
    """The ordered group gather with one store (1024 buckets for it) and with
    the most stores a group takes (16 buckets each): Zipf lookups, the plain
    group gather's bytes and the rows."""
    R, C, N, B = 512, 1024, 500, 300
    stores, slots, tables = [], [], []
    try:
        for t in range(T):
            rb = rows_u8(wl.dlrm_rows(N, R // 4, table=t, seed=21))
            st, sl = _host_store(R, C, rb, host=(t % 3 != 1))
            stores.append(st)
            slots.append(sl)
            tables.append(rb)
        ids = np.stack([wl.zipf_ids(B, N, table=t, seed=22) for t in range(T)], axis=1)
        grp = ibp.ibp_group_create([s.h for s in stores], slots)
        try:
            ref = torch.full((B, T, R), 0xCC, dtype=torch.uint8, device=DEV)
            ibp.ibp_group_gather_decompress(grp, ref, T * R, to_dev(ids), B)
            out = torch.full((B, T, R), 0x33, dtype=torch.uint8, device=DEV)
            ws = torch.empty(ibp.order_workspace_bytes(B * T), dtype=torch.uint8, device=DEV)
            ibp.ibp_group_gather_decompress_ordered(grp, out, T * R, to_dev(ids), B, ws,
                                                    ws.numel())
            for s in stores:
                assert s.status() == ibp.IBP_OK
            assert torch.equal(out, ref)
            o = out.cpu().numpy()
            for t in range(T):
                assert np.array_equal(o[:, t], tables[t][ids[:, t]]), t
        finally:
            ibp.ibp_group_destroy(grp)
    finally:
        for s in stores:
            s.close()


def test_ordered_group_and_packed_decode_in_a_cuda_graph():
    """The ordered group gather (five kernels chained by programmatic
    dependent launch, then the gather) and the packed-cache decode (bulk
    copies on mbarriers) captured once in a CUDA graph and replayed with new
    lookups: every replay returns the rows.  So does a captured plan made
    ahead with its planned gather."""
    R, C, N, B, T = 512, 1024, 3000, 700, 3
    stores, slots, tables = [], [], []
    try:
        for t in range(T):
            rb = rows_u8(wl.dlrm_rows(N, R // 4, table=t, seed=31))
            st, sl = _host_store(R, C, rb, host=(t != 1))
            stores.append(st)
            slots.append(sl)
            tables.append(rb)
        # a packed HBM cache of store 0
        st0 = stores[0]
        stored = torch.zeros(N, dtype=torch.int32, device=DEV)
        d0 = torch.from_numpy(tables[0]).to(DEV)
        s0 = torch.zeros((N, st0.slot), dtype=torch.uint8, device=DEV)
        ibp.ibp_compress(st0.h, s0, d0, R, None, N, stored)
        offs = torch.zeros(N + 1, dtype=torch.int64, device=DEV)
        ibp.ibp_pack(st0.h, None, offs, s0, stored, N)
        cache = torch.zeros(int(offs[-1].item()) + R, dtype=torch.uint8, device=DEV)
        ibp.ibp_pack(st0.h, cache, offs, s0, stored, N)
        grp = ibp.ibp_group_create([s.h for s in stores], slots)
        try:
            ids = torch.zeros((B, T), dtype=torch.int64, device=DEV)
            out = torch.zeros((B, T, R), dtype=torch.uint8, device=DEV)
            ws = torch.empty(ibp.order_workspace_bytes(B * T), dtype=torch.uint8, device=DEV)
            dec = torch.zeros((N, R), dtype=torch.uint8, device=DEV)
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):  # warm-up: launch shapes and store properties known
                ibp.ibp_group_gather_decompress_ordered(grp, out, T * R, ids, B, ws, ws.numel(),
                                                        side)
                ibp.ibp_decompress(st0.h, dec, cache, offs, N, side)
            torch.cuda.synchronize()
            for s in stores:
                assert s.status() == ibp.IBP_OK
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                sp = torch.cuda.current_stream()
                ibp.ibp_group_gather_decompress_ordered(grp, out, T * R, ids, B, ws, ws.numel(),
                                                        sp)
                ibp.ibp_decompress(st0.h, dec, cache, offs, N, sp)
            for step in range(3):
                z = np.stack([wl.zipf_ids(B, N, table=t, seed=40 + step) for t in range(T)],
                             axis=1)
                ids.copy_(torch.from_numpy(z))
                out.zero_()
                dec.zero_()
                g.replay()
                torch.cuda.synchronize()
                for s in stores:
                    assert s.status() == ibp.IBP_OK, step
                o = out.cpu().numpy()
                for t in range(T):
                    assert np.array_equal(o[:, t], tables[t][z[:, t]]), (step, t)
                assert np.array_equal(dec.cpu().numpy(), tables[0]), step
            # a plan made ahead and its gather, captured after one uncaptured pair
            with torch.cuda.stream(side):
                ibp.ibp_group_order_plan(grp, ids, B, ws, ws.numel(), side)
                ibp.ibp_group_gather_decompress_planned(grp, out, T * R, ids, B, ws, ws.numel(),
                                                        side)
            torch.cuda.synchronize()
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2):
                sp = torch.cuda.current_stream()
                ibp.ibp_group_order_plan(grp, ids, B, ws, ws.numel(), sp)
                ibp.ibp_group_gather_decompress_planned(grp, out, T * R, ids, B, ws, ws.numel(),
                                                        sp)
            for step in range(2):
                z = np.stack([wl.zipf_ids(B, N, table=t, seed=50 + step) for t in range(T)],
                             axis=1)
                ids.copy_(torch.from_numpy(z))
                out.zero_()
                g2.replay()
                torch.cuda.synchronize()
                for s in stores:
                    assert s.status() == ibp.IBP_OK, step
                o = out.cpu().numpy()
                for t in range(T):
                    assert np.array_equal(o[:, t], tables[t][z[:, t]]), (step, t)
        finally:
            ibp.ibp_group_destroy(grp)
    finally:
        for s in stores:
            s.close()
