"""GB300-native Invariant Bit Packing (IBP): lossless compression of ML tensors.

The codec runs in hand-written sm_103a CUDA kernels behind a C-ABI library
(``libibp.so``, declared in ``include/ibp.h``).  ``ibp`` is its thin ctypes
binding, ``store.IbpStore`` a torch-facing handle on one store over it;
``workloads`` holds the seeded synthetic inputs.  Importing the
package loads nothing; the binding loads the library on first use and raises
if it has not been built.
"""
__all__ = ["ibp", "store", "workloads"]
