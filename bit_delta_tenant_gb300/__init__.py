"""GB300-native BitDelta hot path: packed 1-bit deltas over a shared bf16 base.

The compute lives in ``libbitdelta.so`` (hand-written sm_103a CUDA behind a
C ABI, declared in ``include/bitdelta.h``).  ``bit_delta_tenant_gb300.bitdelta``
is the thin Python binding with the same entry-point names; ``synth`` makes the
seeded synthetic inputs.  Importing this package loads nothing: the library is
opened on first use and a missing library is an error, never a fallback.
"""
