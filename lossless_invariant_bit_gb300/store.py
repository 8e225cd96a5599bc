"""A torch-facing handle on one IBP store: argument marshalling over ``ibp``.

Every call goes straight to the C-ABI library (``ibp``); this class only
allocates the torch tensors the calls need and passes their pointers.  Rows
are uint8 tensors of shape [n, row_bytes] (any dtype viewed as bytes works
when its rows are contiguous), compressed slots live in pinned host memory
(the zero-copy store of the pages' System Integration) or in HBM.

    st = IbpStore(row_bytes=512, chunk_bytes=1024, n_rows=len(rows))
    st.build(rows_gpu, sample_ids=sample)           # Mask/Bitval from a sample
    slots, stored = st.compress(rows_gpu)           # pinned host slots
    st.set_lengths(stored)                          # optional: one fetch per row
    batch = st.gather(slots, ids_gpu)               # [len(ids), 512] on the GPU
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import torch

from . import ibp


def _bytes2d(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.uint8:
        t = t.reshape(t.shape[0], -1).view(torch.uint8)
    return t


class IbpStore:
    """One store: row geometry, Mask/Bitval and the raw bitmap of its slots."""

    def __init__(self, row_bytes: int, chunk_bytes: int, n_rows: int, slot_bytes: int = 0):
        self.row_bytes, self.chunk_bytes, self.n_rows = row_bytes, chunk_bytes, n_rows
        self.handle = ibp.ibp_store_create(row_bytes, chunk_bytes, n_rows, slot_bytes)
        self.slot_bytes = ibp.ibp_store_get_info(self.handle).slot_bytes
        self._lengths = None  # the attached length table, kept alive while the library reads it

    # -- lifetime
    def close(self) -> None:
        if self.handle:
            ibp.ibp_store_set_lengths(self.handle, None)
            ibp.ibp_store_destroy(self.handle)
            self.handle = None
            self._lengths = None

    def __enter__(self) -> "IbpStore":
        return self

    def __exit__(self, *exc) -> None:
        self.close()

    # -- metadata
    def build(self, rows: torch.Tensor, sample_ids: Optional[torch.Tensor] = None,
              threshold: Tuple[int, int] = (95, 100), stream=None) -> None:
        """Mask/Bitval from rows (all, or the sampled ids) at threshold num/den."""
        rows = _bytes2d(rows)
        n = rows.shape[0] if sample_ids is None else sample_ids.numel()
        ibp.ibp_build_meta(self.handle, rows, rows.stride(0), sample_ids, n, threshold[0],
                           threshold[1], stream)

    def build_tuned(self, rows: torch.Tensor, candidates: Sequence[Tuple[int, int]],
                    sample_ids: Optional[torch.Tensor] = None, stream=None) -> int:
        """Mask/Bitval of the candidate threshold that stores the sample smallest;
        returns its index (synchronises the stream to read it)."""
        rows = _bytes2d(rows)
        n = rows.shape[0] if sample_ids is None else sample_ids.numel()
        chosen = torch.zeros(1, dtype=torch.int32, device=rows.device)
        ibp.ibp_build_meta_tuned(self.handle, rows, rows.stride(0), sample_ids, n,
                                 [c[0] for c in candidates], [c[1] for c in candidates],
                                 chosen, None, stream)
        return int(chosen.item())

    # -- compression
    def compress(self, rows: torch.Tensor, slots: Optional[torch.Tensor] = None,
                 slot_ids: Optional[torch.Tensor] = None, host: bool = True,
                 stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        """Compress rows into slots (allocated when not given: pinned host memory,
        or HBM with host=False).  Returns (slots, stored bytes per row)."""
        rows = _bytes2d(rows)
        if slots is None:
            shape = (self.n_rows, self.slot_bytes)
            slots = (torch.zeros(shape, dtype=torch.uint8, pin_memory=True) if host
                     else torch.zeros(shape, dtype=torch.uint8, device=rows.device))
        stored = torch.empty(rows.shape[0], dtype=torch.int32, device=rows.device)
        ibp.ibp_compress(self.handle, slots, rows, rows.stride(0), slot_ids, rows.shape[0],
                         stored, stream)
        return slots, stored

    def set_lengths(self, stored: Optional[torch.Tensor]) -> None:
        """Attach each slot's stored bytes (the int32 [n_rows] that compress()
        returns, on the device) so that decoders fetch a row's whole stream at
        once; None detaches.  The store keeps a reference while it is attached."""
        if stored is not None and (stored.numel() != self.n_rows or stored.element_size() != 4
                                   or not stored.is_cuda or not stored.is_contiguous()):
            raise ValueError("lengths must be a contiguous 4-byte device tensor of n_rows entries")
        ibp.ibp_store_set_lengths(self.handle, stored)
        self._lengths = stored

    # -- decompression
    def decompress(self, src: torch.Tensor, n: Optional[int] = None,
                   offsets: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                   device=None, stream=None) -> torch.Tensor:
        """Rows 0..n-1 from slots (or a packed cache with its offsets)."""
        n = self.n_rows if n is None else n
        if out is None:
            out = torch.empty((n, self.row_bytes), dtype=torch.uint8,
                              device=device or torch.device("cuda", torch.cuda.current_device()))
        ibp.ibp_decompress(self.handle, out, src, offsets, n, stream)
        return out

    def gather(self, src: torch.Tensor, ids: torch.Tensor, out: Optional[torch.Tensor] = None,
               offsets: Optional[torch.Tensor] = None, ordered: bool = False,
               stream=None) -> torch.Tensor:
        """Rows ids[i] (device int64) from slots or a packed cache, into [len(ids), R].
        ordered=True buckets the ids by address first (for host stores beyond the
        GPU's translation reach, ~20 GB); the rows come out in the same order."""
        n = ids.numel()
        if out is None:
            out = torch.empty((n, self.row_bytes), dtype=torch.uint8, device=ids.device)
        if ordered:
            ws = torch.empty(ibp.order_workspace_bytes(n), dtype=torch.uint8, device=ids.device)
            ibp.ibp_gather_decompress_ordered(self.handle, out, out.stride(0), src, offsets, ids,
                                              n, ws, ws.numel(), stream)
        else:
            ibp.ibp_gather_decompress(self.handle, out, src, offsets, ids, n, stream)
        return out

    def pack(self, slots: torch.Tensor, stored: torch.Tensor,
             stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        """A packed HBM cache of the slots: (cache bytes, offsets[n + 1])."""
        n = stored.numel()
        offsets = torch.zeros(n + 1, dtype=torch.int64, device=stored.device)
        ibp.ibp_pack(self.handle, None, offsets, slots, stored, n, stream)
        total = int(offsets[-1].item())
        cache = torch.zeros(total + self.row_bytes, dtype=torch.uint8, device=stored.device)
        ibp.ibp_pack(self.handle, cache, offsets, slots, stored, n, stream)
        return cache, offsets

    def status(self, reset: bool = True) -> int:
        """The store's device status word (synchronises the device)."""
        return ibp.ibp_stream_status(self.handle, reset=reset)
