"""CPU oracle for Invariant Bit Packing (IBP) -- TEST INFRASTRUCTURE ONLY.

Two independent restatements of the format: ``ibp_ref`` (pure Python, small
inputs) and ``ibp_ref.c`` (plain C, loaded through ``ref_c``).  Only the test
suite, the smoke check and the benchmark's CPU-baseline leg use this package.
The GPU library neither imports nor calls it, and it shares no code with the
GPU library.
"""
