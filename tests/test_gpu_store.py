"""IbpStore (the torch-facing handle): a round trip through every call it
wraps, checked against the rows and the oracle's stored sizes."""
import numpy as np
import pytest
import torch

from lossless_invariant_bit_gb300 import ibp
from lossless_invariant_bit_gb300 import workloads as wl
from lossless_invariant_bit_gb300.store import IbpStore
from oracle import ref_c

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.mark.parametrize("host", [True, False])
def test_store_round_trip(host):
    n = 5000
    rows = wl.dense_gnn_rows(n, seed=21)               # fp32 [n, 128]
    d = torch.from_numpy(rows).to(DEV)                 # passed as fp32: viewed as bytes
    sample = torch.from_numpy(wl.sample_ids(n, 50, seed=21)).to(DEV)
    rb = rows.view(np.uint8)
    with IbpStore(512, 256, n) as st:
        st.build(d, sample_ids=sample)
        slots, stored = st.compress(d, host=host)
        m = np.zeros(128, np.uint32)
        b = np.zeros(128, np.uint32)
        ibp.ibp_meta_get(st.handle, m, b)
        mr, br = ref_c.build_meta(rb, 95, 100, sample_ids=sample.cpu().numpy())
        assert np.array_equal(m, mr) and np.array_equal(b, br)
        ref_st = ref_c.compress_batch(rb, 256, mr, br, np.zeros((n, 512), np.uint8),
                                      np.zeros((n + 31) // 32, np.uint32), nthreads=8)
        assert np.array_equal(stored.cpu().numpy().astype(np.uint32), ref_st)
        assert np.array_equal(st.decompress(slots).cpu().numpy(), rb)
        ids = torch.from_numpy(wl.uniform_ids(3 * n, n, seed=2)).to(DEV)
        got = st.gather(slots, ids)
        assert np.array_equal(got.cpu().numpy(), rb[ids.cpu().numpy()])
        assert torch.equal(st.gather(slots, ids, ordered=True), got)
        st.set_lengths(stored)  # whole-stream fetches: same rows
        assert torch.equal(st.gather(slots, ids), got)
        assert torch.equal(st.gather(slots, ids, ordered=True), got)
        st.set_lengths(None)
        with pytest.raises(ValueError):
            st.set_lengths(stored[:-1])
        cache, offs = st.pack(slots.to(DEV) if host else slots, stored)
        assert np.array_equal(st.gather(cache, ids, offsets=offs[:-1]).cpu().numpy(),
                              rb[ids.cpu().numpy()])
        assert st.status() == ibp.IBP_OK


def test_store_tuned_build_picks_cheapest():
    n = 20000
    rows = torch.from_numpy(wl.sparse_gnn_rows(n, seed=3)).to(DEV)
    cands = [(95, 100), (999, 1000), (1, 1)]
    with IbpStore(512, 1024, n) as st:
        k = st.build_tuned(rows, cands)
        assert cands[k] == (999, 1000)  # the sparse rows' 7 exponent bits stay: 116 B rows
        _, stored = st.compress(rows, host=False)
        assert int(stored.max().item()) <= 116
