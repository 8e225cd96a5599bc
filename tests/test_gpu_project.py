"""The K/V projection with the compressor in its epilogue
(ibp_project_compress) against the oracle.

The projection Y = X W^T (+ bias) runs on the tensor cores with fp32
accumulation and rounds to 16 bits; a plain fp32 reference of the same
product sums in another order, so Y is checked against the reference within
the bound of fp32 summation error plus one unit in the last place (and
nearly all values must agree exactly).  The compressed rows, raw bits and stored sizes are
checked bit for bit against the oracle's compression of the kernel's own Y
(the float arithmetic decides Y; the rest is integer work on Y).  Inputs are
K/V-shaped: per output channel a log-normal scale with a few outlier
channels, as the KV workload's channels have."""
import numpy as np
import pytest
import torch

from lossless_invariant_bit_gb300 import ibp
from oracle import ref_c
from tests.gpu_util import DEV, Store, assert_streams_equal

pytestmark = pytest.mark.gpu


def _weights(N, K, dtype, seed, outliers=0.02):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    scale = torch.exp(0.5 * torch.randn(N, generator=g, device=DEV))
    oc = torch.randperm(N, generator=g, device=DEV)[:max(1, int(outliers * N))]
    scale[oc] *= 20.0
    w = (torch.randn((N, K), generator=g, device=DEV) * (scale[:, None] / K ** 0.5)).to(dtype)
    b = (torch.randn(N, generator=g, device=DEV) * 0.1 * scale).to(dtype)
    return w, b


def _within_bound(y: torch.Tensor, x: torch.Tensor, w: torch.Tensor, ref: torch.Tensor):
    """Both Y and the reference are fp32 dot products of length K rounded to
    16 bits.  Each fp32 sum is within g_K * sum_k |x_k w_k| of the exact one,
    g_K = K u / (1 - K u), u = 2^-24 (recursive summation in any order), so
    the two sums differ by at most 2 g_K sum |x w|, and after rounding the
    16-bit values by at most that plus one unit in the last place of the
    reference.  Returns (bound met everywhere, fraction exactly equal)."""
    K = x.shape[1]
    u = 2.0 ** -24
    gk = K * u / (1 - K * u)
    absdot = x.float().abs() @ w.float().abs().T
    r = ref.abs()
    ulp = (r.view(torch.int16) + 1).view(ref.dtype).float() - r.float()
    err = (y.float() - ref.float()).abs()
    ok = bool((err <= ulp + 2 * gk * absdot).all())
    return ok, float((y.view(torch.int16) == ref.view(torch.int16)).float().mean())


def _run(st, x, w, b, dtype_code, slots, slot_ids=None, stream=None):
    m, K = x.shape
    N = w.shape[0]
    y = torch.empty((m, N), dtype=x.dtype, device=DEV)
    stored = torch.full((m,), -1, dtype=torch.int32, device=DEV)
    wsb = ibp.project_workspace_bytes(m, 2 * N)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    ibp.ibp_project_compress(st.h, x, m, K, w, b, dtype_code, y, slots, slot_ids, stored, ws, wsb,
                             stream)
    torch.cuda.synchronize()
    return y, stored.cpu().numpy().astype(np.uint32)


def _check_against_oracle(st, y, stored, slots, slot_ids_np, R, C=256):
    m = y.shape[0]
    yb = y.contiguous().view(torch.uint8).cpu().numpy().reshape(m, R)
    mask, bitval = st.meta()
    ref_sl = np.zeros((m, st.slot), np.uint8)
    ref_bm = np.zeros((m + 31) // 32, np.uint32)
    ref_st = ref_c.compress_batch(yb, C, mask, bitval, ref_sl, ref_bm, nthreads=8)
    assert np.array_equal(stored, ref_st)
    sl = slots.cpu().numpy() if slots.device.type == "cuda" else slots.numpy()
    ids = np.arange(m) if slot_ids_np is None else slot_ids_np
    assert_streams_equal(sl[ids], ref_sl, ref_st, rows=ids)
    bm = st.bitmap()
    for j, i in enumerate(ids):
        assert (bm[i >> 5] >> (i & 31)) & 1 == (ref_bm[j >> 5] >> (j & 31)) & 1, i
    return yb


@pytest.mark.parametrize("m,K,dtype,bias", [
    (20, 4096, torch.float16, True),    # a decode step of one (layer, K|V): OPT-6.7B shape
    (300, 512, torch.float16, False),   # three row tiles, the last one ragged
    (20, 64, torch.bfloat16, True),     # one K block, bf16
    (129, 4096, torch.bfloat16, False),  # a tile and one row
])
def test_project_compress_matches_reference_and_oracle(m, K, dtype, bias):
    N, R = 4096, 8192
    code = 1 if dtype == torch.bfloat16 else 0
    w, b = _weights(N, K, dtype, seed=m * 7 + K)
    b = b if bias else None
    g = torch.Generator(device=DEV)
    g.manual_seed(m + K)
    # the Mask/Bitval from "prompt" rows of the same projection
    xp = torch.randn((512, K), generator=g, device=DEV).to(dtype)
    yp = xp.float() @ w.float().T
    if b is not None:
        yp += b.float()
    yp = yp.to(dtype).contiguous()
    n_rows = 4 * m + 64
    st = Store(R, 256, n_rows, R)
    try:
        ibp.ibp_build_meta(st.h, yp.view(torch.uint8), R, None, 512, 95, 100)
        x = torch.randn((m, K), generator=g, device=DEV).to(dtype)
        slots = torch.zeros((n_rows, R), dtype=torch.uint8, pin_memory=True)
        sid_np = (np.arange(m, dtype=np.int64) * 3 + 5)
        sid = torch.from_numpy(sid_np).to(DEV)
        y, stored = _run(st, x, w, b, code, slots, sid)
        assert st.status() == ibp.IBP_OK
        ref = x.float() @ w.float().T
        if b is not None:
            ref += b.float()
        ref = ref.to(dtype)
        ok, exact = _within_bound(y, x, w, ref)
        assert ok, "projection outside the fp32 summation bound"
        assert exact > 0.9  # most values round identically; the bound above is the test
        _check_against_oracle(st, y, stored, slots, sid_np, R)
        # the rows decode back to Y
        out = torch.empty((m, R), dtype=torch.uint8, device=DEV)
        ibp.ibp_gather_decompress(st.h, out, slots, None, sid, m)
        assert st.status() == ibp.IBP_OK
        assert torch.equal(out, y.contiguous().view(torch.uint8).view(m, R))
        # some chunks pack and some rows carry raw chunks, as K/V rows do
        assert (stored < R).any()
    finally:
        st.close()


def test_project_compress_all_raw_store_and_bad_slot():
    """A store with no Mask yet stores every row raw; a slot id out of range
    sets IBP_ERANGE and leaves the other rows correct."""
    m, K, N, R = 40, 256, 512, 1024
    w, b = _weights(N, K, torch.float16, seed=3)
    st = Store(R, 256, 64, R)
    try:
        x = torch.randn((m, K), device=DEV).to(torch.float16)
        slots = torch.zeros((64, R), dtype=torch.uint8, device=DEV)
        y, stored = _run(st, x, w, b, 0, slots)
        assert st.status() == ibp.IBP_OK
        assert (stored == R).all()
        assert np.array_equal(slots[:m].cpu().numpy(),
                              y.contiguous().view(torch.uint8).cpu().numpy().reshape(m, R))
        sid_np = np.arange(m, dtype=np.int64)
        sid_np[7] = 64  # out of range
        sid = torch.from_numpy(sid_np).to(DEV)
        slots.zero_()
        y, stored = _run(st, x, w, b, 0, slots, sid)
        assert st.status() == ibp.IBP_ERANGE
        assert stored[7] == 0
        ok = np.delete(np.arange(m), 7)
        assert np.array_equal(slots[ok].cpu().numpy(),
                              y.contiguous().view(torch.uint8).cpu().numpy().reshape(m, R)[ok])
    finally:
        st.close()


def test_project_compress_rejects_bad_geometry():
    st = Store(8192, 1024, 64, 8192)  # chunks of 1 KB: not one 128-column tile
    try:
        x = torch.zeros((4, 64), dtype=torch.float16, device=DEV)
        w = torch.zeros((4096, 64), dtype=torch.float16, device=DEV)
        y = torch.empty((4, 4096), dtype=torch.float16, device=DEV)
        slots = torch.zeros((64, 8192), dtype=torch.uint8, device=DEV)
        ws = torch.empty(ibp.project_workspace_bytes(4, 8192), dtype=torch.uint8, device=DEV)
        with pytest.raises(ibp.IbpError) as e:
            ibp.ibp_project_compress(st.h, x, 4, 64, w, None, 0, y, slots, None, None, ws,
                                     ws.numel())
        assert e.value.status == ibp.IBP_EINVAL
    finally:
        st.close()
    st = Store(8192, 256, 64, 8192)
    try:
        with pytest.raises(ibp.IbpError) as e:  # k_dim not a multiple of 64
            ibp.ibp_project_compress(st.h, x, 4, 48, w, None, 0, y, slots, None, None, ws,
                                     ws.numel())
        assert e.value.status == ibp.IBP_EINVAL
        with pytest.raises(ibp.IbpError) as e:  # short workspace
            ibp.ibp_project_compress(st.h, x, 4, 64, w, None, 0, y, slots, None, None, ws, 64)
        assert e.value.status == ibp.IBP_EINVAL
    finally:
        st.close()


def test_project_compress_captured_in_a_cuda_graph():
    """A decode step's projection captured once in a CUDA graph (the two
    kernels, the second launched behind the first) and replayed with new
    inputs: every replay writes the bytes an uncaptured call writes for the
    same inputs (Y, stored bytes, sizes, raw bits)."""
    m, K, N, R = 20, 4096, 4096, 8192
    dtype = torch.float16
    w, b = _weights(N, K, dtype, seed=77)
    g = torch.Generator(device=DEV)
    g.manual_seed(78)
    xp = torch.randn((512, K), generator=g, device=DEV).to(dtype)
    yp = (xp.float() @ w.float().T + b.float()).to(dtype).contiguous()
    n_rows = 64
    st = Store(R, 256, n_rows, R)
    try:
        ibp.ibp_build_meta(st.h, yp.view(torch.uint8), R, None, 512, 95, 100)
        x = torch.zeros((m, K), dtype=dtype, device=DEV)
        y = torch.empty((m, N), dtype=dtype, device=DEV)
        slots = torch.zeros((n_rows, R), dtype=torch.uint8, device=DEV)
        stored = torch.zeros(m, dtype=torch.int32, device=DEV)
        wsb = ibp.project_workspace_bytes(m, R)
        ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # warm-up: kernel limits set, store properties known
            ibp.ibp_project_compress(st.h, x, m, K, w, b, 0, y, slots, None, stored, ws, wsb, side)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            ibp.ibp_project_compress(st.h, x, m, K, w, b, 0, y, slots, None, stored, ws, wsb,
                                     torch.cuda.current_stream())
        for step in range(3):
            xs = torch.randn((m, K), generator=g, device=DEV).to(dtype)
            x.copy_(xs)
            slots.zero_()
            gr.replay()
            torch.cuda.synchronize()
            assert st.status() == ibp.IBP_OK
            got = (y.clone(), slots[:m].clone(), stored.clone(), st.bitmap().copy())
            slots.zero_()
            ibp.ibp_project_compress(st.h, xs, m, K, w, b, 0, y, slots, None, stored, ws, wsb)
            torch.cuda.synchronize()
            assert st.status() == ibp.IBP_OK
            assert torch.equal(got[0], y), step
            assert torch.equal(got[1], slots[:m]), step
            assert torch.equal(got[2], stored), step
            assert np.array_equal(got[3], st.bitmap()), step
    finally:
        st.close()
