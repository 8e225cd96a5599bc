"""The pages' workloads end to end on the GPU, at reduced sizes, against the
oracle: dense GNN (2-hop mini-batch, chunk sweep), DLRM (26 tables, Zipf
lookups, strided [batch, tables, dim] output) and the KV-cache flow (meta
from prompt rows, per-token compression at decode, per-layer re-fetch).
"""
import numpy as np
import pytest
import torch

from lossless_invariant_bit_gb300 import ibp
from lossless_invariant_bit_gb300 import workloads as wl
from oracle import ref_c
from tests.gpu_util import DEV, Store, assert_streams_equal, oracle_slots, rows_u8

pytestmark = pytest.mark.gpu


def _host_store(st, rows_b, sample=None, num=95, den=100):
    """Build meta on the GPU from (sampled) rows and compress all rows into
    pinned host slots.  Returns (slots, stored sizes)."""
    n, R = rows_b.shape
    d = torch.from_numpy(rows_b).to(DEV)
    ids = None if sample is None else torch.from_numpy(sample).to(DEV)
    ibp.ibp_build_meta(st.h, d, R, ids, n if sample is None else len(sample), num, den)
    slots = torch.empty((n, st.slot), dtype=torch.uint8, pin_memory=True)
    stored = torch.empty(n, dtype=torch.int32, device=DEV)
    ibp.ibp_compress(st.h, slots, d, R, None, n, stored)
    torch.cuda.synchronize()
    assert st.status() == ibp.IBP_OK
    return slots, stored.cpu().numpy().astype(np.uint32)


@pytest.mark.parametrize("C", [256, 1024, 4096])
def test_dense_gnn_two_hop(C):
    n_rows = 200_000
    rows = wl.dense_gnn_rows(n_rows, seed=0)
    rb = rows_u8(rows)
    sample = wl.sample_ids(n_rows, 10, seed=0)
    st = Store(512, C, n_rows)
    try:
        slots, stored = _host_store(st, rb, sample)
        m, b = st.meta()
        mr, br = ref_c.build_meta(rb, 95, 100, sample_ids=sample)
        assert np.array_equal(m, mr) and np.array_equal(b, br)
        pick = np.random.default_rng(C).choice(n_rows, 5000, replace=False)
        ref_sl, _, ref_st = oracle_slots(rb[pick], C, mr, br, st.slot)
        assert np.array_equal(stored[pick], ref_st)
        assert_streams_equal(slots.numpy()[pick], ref_sl, ref_st, rows=pick)
        ratio = stored.sum() / (n_rows * 512)
        assert 0.80 < ratio < 0.95  # modest saving, as the pages report for dense GNN
        ids = wl.two_hop_ids(n_rows, seed=1)
        d_ids = torch.from_numpy(ids).to(DEV)
        out = torch.empty((len(ids), 512), dtype=torch.uint8, device=DEV)
        ibp.ibp_gather_decompress(st.h, out, slots, None, d_ids, len(ids))
        assert st.status() == ibp.IBP_OK
        assert np.array_equal(out.cpu().numpy(), rb[ids])
        # the same store as an HBM cache (slot layout): the fast decoder's path
        info = ibp.ibp_store_get_info(st.h)
        assert info.max_runs <= 2
        out.zero_()
        ibp.ibp_gather_decompress(st.h, out, slots.to(DEV), None, d_ids, len(ids))
        assert st.status() == ibp.IBP_OK
        assert np.array_equal(out.cpu().numpy(), rb[ids])
    finally:
        st.close()


def test_dense_gnn_chunk_1k_equals_4k():
    """C >= R means one chunk per 512 B row, so 1 KB and 4 KB chunks give the
    same stream for every row (one of the format's readings)."""
    n_rows = 50_000
    rb = rows_u8(wl.dense_gnn_rows(n_rows, seed=2))
    sample = wl.sample_ids(n_rows, 10, seed=2)
    res = []
    for C in (1024, 4096):
        st = Store(512, C, n_rows)
        try:
            slots, stored = _host_store(st, rb, sample)
            res.append((stored, slots.numpy().copy(), st.bitmap()))
        finally:
            st.close()
    (s1, sl1, b1), (s2, sl2, b2) = res
    assert np.array_equal(s1, s2) and np.array_equal(b1, b2)
    for i in range(0, n_rows, 97):
        assert np.array_equal(sl1[i, :s1[i]], sl2[i, :s2[i]])


@pytest.mark.parametrize("dim", [128, 256, 512])
def test_dlrm_26_tables_strided(dim):
    T, n_rows, B, R, C = 26, 20_000, 8192, dim * 4, 1024
    out = torch.full((B, T, R), 0xEE, dtype=torch.uint8, device=DEV)
    want = np.empty((B, T, R), np.uint8)
    for t in range(T):
        rows = wl.dlrm_rows(n_rows, dim, table=t, seed=0)
        rb = rows_u8(rows)
        sample = wl.sample_ids(n_rows, 10, seed=t)
        st = Store(R, C, n_rows)
        try:
            slots, stored = _host_store(st, rb, sample)
            if t % 13 == 0:
                m, b = st.meta()
                mr, br = ref_c.build_meta(rb, 95, 100, sample_ids=sample)
                assert np.array_equal(m, mr) and np.array_equal(b, br)
                ref_sl, _, ref_st = oracle_slots(rb[:3000], C, mr, br, st.slot)
                assert np.array_equal(stored[:3000], ref_st)
                assert_streams_equal(slots.numpy()[:3000], ref_sl, ref_st)
            ids = wl.zipf_ids(B, n_rows, table=t, seed=0)
            src = slots if t % 2 == 0 else slots.to(DEV)  # host link or HBM cache
            ibp.ibp_gather_decompress_strided(st.h, out[:, t], T * R, src, None,
                                              torch.from_numpy(ids).to(DEV), B)
            assert st.status() == ibp.IBP_OK
            want[:, t] = rb[ids]
        finally:
            st.close()
    assert np.array_equal(out.cpu().numpy(), want)


def test_kv_cache_prefill_decode_flow():
    """Per (layer, K|V): Mask/Bitval from all prompt rows (prefill), prompt rows
    compressed into host slots, then at each decode step the new token's row is
    compressed on the GPU into its slot and the layer's history is re-fetched."""
    layers, batch, prompt, steps, seq = 2, 3, 96, 4, 128
    R, C = 4096 * 2, 256
    for layer in range(layers):
        for kv in range(2):
            sc = wl.kv_channel_scales(layer, kv)
            full = wl.kv_rows(layer, kv, batch, range(prompt + steps), scales=sc)
            fb = full.view(np.uint8).reshape(batch, prompt + steps, R)
            st = Store(R, C, batch * seq)
            try:
                prompt_rows = np.ascontiguousarray(fb[:, :prompt]).reshape(-1, R)
                d_prompt = torch.from_numpy(prompt_rows).to(DEV)
                ibp.ibp_build_meta(st.h, d_prompt, R, None, len(prompt_rows), 95, 100)
                m, b = st.meta()
                mr, br = ref_c.build_meta(prompt_rows, 95, 100)
                assert np.array_equal(m, mr) and np.array_equal(b, br)
                slots = torch.zeros((batch * seq, st.slot), dtype=torch.uint8, pin_memory=True)
                pid = wl.kv_row_ids(batch, prompt, seq)
                stored = torch.empty(len(pid), dtype=torch.int32, device=DEV)
                ibp.ibp_compress(st.h, slots, d_prompt, R, torch.from_numpy(pid).to(DEV),
                                 len(pid), stored)
                for s in range(steps):
                    tok = np.ascontiguousarray(fb[:, prompt + s])
                    sid = np.arange(batch, dtype=np.int64) * seq + prompt + s
                    st_tok = torch.empty(batch, dtype=torch.int32, device=DEV)
                    ibp.ibp_compress(st.h, slots, torch.from_numpy(tok).to(DEV), R,
                                     torch.from_numpy(sid).to(DEV), batch, st_tok)
                    ref_sl, _, ref_st = oracle_slots(tok, C, mr, br, st.slot)
                    torch.cuda.synchronize()
                    assert np.array_equal(st_tok.cpu().numpy().astype(np.uint32), ref_st)
                    assert_streams_equal(slots.numpy()[sid], ref_sl, ref_st)
                    hist = wl.kv_row_ids(batch, prompt + s + 1, seq)
                    out = torch.empty((len(hist), R), dtype=torch.uint8, device=DEV)
                    ibp.ibp_gather_decompress(st.h, out, slots, None,
                                              torch.from_numpy(hist).to(DEV), len(hist))
                    assert st.status() == ibp.IBP_OK
                    want = fb[:, :prompt + s + 1].reshape(-1, R)
                    assert np.array_equal(out.cpu().numpy(), want)
            finally:
                st.close()


@pytest.mark.parametrize("R,C", [(4096, 256), (4096, 1024), (4096, 4096), (1024, 256)])
@pytest.mark.parametrize("k", [0, 4, 16, 28])
@pytest.mark.parametrize("scattered", [False, True])
def test_space_saving_sweep_rows(R, C, k, scattered):
    """The space-saving sweep's input at reduced size: the GPU builder and
    compressor agree with the oracle, and the gather from host slots returns
    the rows, at every saving and chunk size of the sweep."""
    n = 3000 if R == 4096 else 6000
    rb = wl.invariant_rows(n, R, k, scattered, seed=2)
    sample = wl.sample_ids(n, 100, seed=2)
    st = Store(R, C, n)
    try:
        slots, stored = _host_store(st, rb, sample)
        mr, br = ref_c.build_meta(rb, 95, 100, sample_ids=sample)
        m, b = st.meta()
        assert np.array_equal(m, mr) and np.array_equal(b, br)
        ref_sl, ref_bm, ref_st = oracle_slots(rb, C, mr, br, st.slot)
        assert np.array_equal(stored, ref_st)
        assert np.array_equal(st.bitmap(), ref_bm)
        assert_streams_equal(slots.numpy(), ref_sl, ref_st)
        ids = wl.uniform_ids(2 * n, n, seed=3)
        out = torch.empty((len(ids), R), dtype=torch.uint8, device=DEV)
        ibp.ibp_gather_decompress(st.h, out, slots, None, torch.from_numpy(ids).to(DEV), len(ids))
        assert st.status() == ibp.IBP_OK
        assert np.array_equal(out.cpu().numpy(), rb[ids])
    finally:
        st.close()


@pytest.mark.parametrize("R,C,H", [(8192, 256, 32), (1024, 128, 8), (2048, 512, 4)])
def test_kv_fetch_into_attention_layout(R, C, H):
    """ibp_gather_decompress_split: K rows of B sequences (one token = H heads
    of D fp16, chunk = one head) land in a [B, H, T, D] tensor; a raw row, an
    out-of-range id (zeros) and the padding between sequences (untouched)."""
    D = R // (2 * H)
    assert C == 2 * D
    B, T_store, T = 3, 64, 41
    rows = wl.kv_rows(2, 0, B, range(T_store), channels=R // 2, seed=4)  # [B, T_store, R/2] fp16
    rb = rows.view(np.uint8).reshape(B * T_store, R).copy()
    rb[5] = np.random.default_rng(0).integers(0, 256, R, dtype=np.uint8)  # an incompressible row
    st = Store(R, C, B * T_store)
    try:
        prompt = (np.arange(B)[:, None] * T_store + np.arange(32)[None, :]).reshape(-1)
        slots, stored = _host_store(st, rb, prompt)
        ids = (np.arange(B)[:, None] * T_store + np.arange(T)[None, :]).reshape(-1).astype(np.int64)
        ids[7] = B * T_store + 3  # out of range: its pieces are zeroed
        gpad = 4096  # bytes between sequences, left untouched
        gstride = H * T * D * 2 + gpad
        out = torch.full((B * gstride,), 0xCC, dtype=torch.uint8, device=DEV)
        ibp.ibp_gather_decompress_split(st.h, out, T, gstride, D * 2, T * D * 2, slots, None,
                                        torch.from_numpy(ids).to(DEV), len(ids))
        assert st.status() == ibp.IBP_ERANGE
        o = out.cpu().numpy().reshape(B, gstride)
        got = o[:, :H * T * D * 2].reshape(B, H, T, D * 2)
        want = rb[np.clip(ids, 0, B * T_store - 1)].reshape(B, T, H, D * 2).transpose(0, 2, 1, 3)
        want = want.copy()
        want[0, :, 7] = 0
        assert np.array_equal(got, want)
        assert np.all(o[:, H * T * D * 2:] == 0xCC)
        # the same rows through the plain gather, transposed on the host
        ids_ok = ids.copy()
        ids_ok[7] = 0
        flat = torch.empty((len(ids), R), dtype=torch.uint8, device=DEV)
        ibp.ibp_gather_decompress(st.h, flat, slots, None, torch.from_numpy(ids_ok).to(DEV),
                                  len(ids))
        assert st.status() == ibp.IBP_OK
        f = flat.cpu().numpy().reshape(B, T, H, D * 2).transpose(0, 2, 1, 3)
        mask = np.ones((B, H, T), bool)
        mask[0, :, 7] = False
        assert np.array_equal(f[mask], got[mask])
    finally:
        st.close()


def test_split_gather_rejects_other_geometries():
    a = Store(1000 // 16 * 16, 100, 16)  # chunk of 100 B: not whole 16-byte groups
    b = Store(16384, 1024, 16)           # rows above 8 KB
    try:
        ids = torch.zeros(4, dtype=torch.int64, device=DEV)
        buf = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
        for s in (a, b):
            with pytest.raises(ibp.IbpError) as e:
                ibp.ibp_gather_decompress_split(s.h, buf, 4, 0, 16, 256, buf, None, ids, 4)
            assert e.value.status == ibp.IBP_EINVAL
        c = Store(1024, 256, 16)
        try:
            with pytest.raises(ibp.IbpError) as e:  # strides must be multiples of 16
                ibp.ibp_gather_decompress_split(c.h, buf, 4, 0, 8, 256, buf, None, ids, 4)
            assert e.value.status == ibp.IBP_EALIGN
        finally:
            c.close()
    finally:
        a.close()
        b.close()


def test_bf16_weight_offload_stream():
    """bf16 weight matrices (the weight-offload stream): the GPU builder and
    compressor match the oracle, the dense decompression from host slots
    returns the weights, and the saving is of the order the pages report."""
    R, C, n = 8192, 256, 700
    try_stores = []
    try:
        for m in range(2):
            rb = wl.bf16_weight_rows(n, 4096, seed=5, matrix=m).view(np.uint8).reshape(n, R)
            sample = wl.sample_ids(n, 100, seed=m)
            st = Store(R, C, n)
            try_stores.append(st)
            slots, stored = _host_store(st, rb, sample)
            mr, br = ref_c.build_meta(rb, 95, 100, sample_ids=sample)
            mm, bb = st.meta()
            assert np.array_equal(mm, mr) and np.array_equal(bb, br)
            ref_sl, ref_bm, ref_st = oracle_slots(rb, C, mr, br, st.slot)
            assert np.array_equal(stored, ref_st)
            assert_streams_equal(slots.numpy(), ref_sl, ref_st)
            assert 0.70 < stored.sum() / rb.size < 0.90
            out = torch.empty((n, R), dtype=torch.uint8, device=DEV)
            ibp.ibp_decompress(st.h, out, slots, None, n)
            assert st.status() == ibp.IBP_OK
            assert np.array_equal(out.cpu().numpy(), rb)
    finally:
        for st in try_stores:
            st.close()


def test_decode_step_captured_in_a_cuda_graph():
    """A KV decode step (compress the step's new rows into their slots, then
    gather the history) captured once in a CUDA graph and replayed with new
    rows: every replay's gather returns the rows it just compressed."""
    R, C, B, T = 8192, 256, 4, 96
    N = B * T
    rows = wl.kv_rows(1, 1, B, range(T), seed=9).view(np.uint8).reshape(N, R)
    st = Store(R, C, N)
    try:
        prompt = (np.arange(B)[:, None] * T + np.arange(64)[None, :]).reshape(-1)
        slots, _ = _host_store(st, rows, prompt)
        new = torch.zeros((B, R), dtype=torch.uint8, device=DEV)
        sids = torch.zeros(B, dtype=torch.int64, device=DEV)
        ids = torch.from_numpy(np.arange(N, dtype=np.int64)).to(DEV)
        out = torch.zeros((N, R), dtype=torch.uint8, device=DEV)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # warm-up: store properties and launch shapes known
            ibp.ibp_compress(st.h, slots, new, R, sids, B, None, side)
            ibp.ibp_gather_decompress(st.h, out, slots, None, ids, N, side)
        torch.cuda.synchronize()
        ibp.ibp_compress(st.h, slots, torch.from_numpy(rows[:B]).to(DEV), R,
                         torch.arange(B, dtype=torch.int64, device=DEV), B, None)
        torch.cuda.synchronize()
        assert st.status() == ibp.IBP_OK
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            sp = torch.cuda.current_stream()
            ibp.ibp_compress(st.h, slots, new, R, sids, B, None, sp)
            ibp.ibp_gather_decompress(st.h, out, slots, None, ids, N, sp)
        expect = rows.copy()
        gen = np.random.default_rng(11)
        for step in range(3):
            t = 64 + step
            tok = (np.arange(B) * T + t).astype(np.int64)
            fresh = wl.kv_rows(1, 1, B, [T + 100 + step], seed=9).view(np.uint8).reshape(B, R).copy()
            fresh[gen.integers(0, B)] = gen.integers(0, 256, R, dtype=np.uint8)  # one raw row
            new.copy_(torch.from_numpy(fresh))
            sids.copy_(torch.from_numpy(tok))
            g.replay()
            torch.cuda.synchronize()
            assert st.status() == ibp.IBP_OK
            expect[tok] = fresh
            assert np.array_equal(out.cpu().numpy(), expect), step
    finally:
        st.close()


def test_graph_replayed_after_a_rebuild_reports_einval():
    """A decompression and a compression captured in a CUDA graph keep the
    store properties of the Mask/Bitval current at capture.  Replayed after
    the Mask/Bitval was rebuilt, they must not decode or pack with them: the
    decompression zero-fills its rows and the compression writes nothing,
    both setting IBP_EINVAL.  A fresh capture works again."""
    rows, _ = wl.tiny_rows(seed=21, n_rows=2048, raw_frac=0.01)
    rb = rows_u8(rows)
    n, R, C = rb.shape[0], rb.shape[1], 256
    st = Store(R, C, n, R)
    try:
        d = torch.from_numpy(rb).to(DEV)
        ibp.ibp_build_meta(st.h, d, R, None, n, 95, 100)
        slots = torch.zeros((n, R), dtype=torch.uint8, device=DEV)
        ibp.ibp_compress(st.h, slots, d, R, None, n, None)
        torch.cuda.synchronize()  # the store's properties reach the host
        out = torch.zeros((n, R), dtype=torch.uint8, device=DEV)
        slots2 = torch.zeros_like(slots)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # warm-up of the specialised forms
            ibp.ibp_decompress(st.h, out, slots, None, n, side)
            ibp.ibp_compress(st.h, slots2, d, R, None, n, None, side)
        torch.cuda.synchronize()
        assert st.status() == ibp.IBP_OK
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            sp = torch.cuda.current_stream()
            ibp.ibp_decompress(st.h, out, slots, None, n, sp)
            ibp.ibp_compress(st.h, slots2, d, R, None, n, None, sp)
        out.zero_()
        slots2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert st.status() == ibp.IBP_OK
        assert np.array_equal(out.cpu().numpy(), rb)
        assert torch.equal(slots2, slots)
        # a rebuild (another threshold) starts a new generation of the store's tables
        ibp.ibp_build_meta(st.h, d, R, None, n, 1, 1)
        torch.cuda.synchronize()
        out.fill_(0x5A)
        slots2.fill_(0x77)
        g.replay()
        torch.cuda.synchronize()
        assert st.status() == ibp.IBP_EINVAL
        assert not out.any(), "stale replay must zero-fill its rows"
        assert bool((slots2 == 0x77).all()), "stale replay must not write slots"
        # uncaptured calls and a new capture use the new tables
        ibp.ibp_compress(st.h, slots, d, R, None, n, None)
        torch.cuda.synchronize()
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2):
            ibp.ibp_decompress(st.h, out, slots, None, n, torch.cuda.current_stream())
        g2.replay()
        torch.cuda.synchronize()
        assert st.status() == ibp.IBP_OK
        assert np.array_equal(out.cpu().numpy(), rb)
    finally:
        st.close()
