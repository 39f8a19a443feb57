"""Persistent batch-1 decode megakernel for GB300 (sm_103a).

`mbk` is the ctypes binding of the C-ABI library (libmbk.so, built from csrc/); `workloads`
draws seeded synthetic decoders and token streams.
"""
