"""CPU oracle for segment-causal KV-cache attention (test infrastructure only).

This package is the plain, slow, obviously correct reference that the CUDA path
is checked against.  It is NOT part of the product: only the test suite, the
``smoke()`` entry point and the benchmark's CPU-baseline leg may import it.  It
shares no code with the CUDA library and never imports it.

Precision: float64 for everything except the INT8 codec, whose bits are defined
in IEEE float32 so that GPU codes and scales can be compared bit for bit.

Modules
-------
rope3d       3D rotary position embedding over (latent frame, h, w)
int8_codec   per-(token, head) absmax INT8 quantisation of K/V rows
ring_cache   the persistent, optionally windowed ring of latent frames
attention    segment attention over [resident cache ; current segment] and the
             equivalent full-sequence masked formulation
sparse       block-sparse variant: per query group, the highest-scoring cache
             key tiles plus all current keys

Parity status: every function here is pinned by the ``tests/test_oracle_*``
suite (closed forms, invariants, brute force and the pages' printed numbers),
except the RoPE pairing convention and the text-token positions, which the
pages leave open; those two readings are "parity unpinned" beyond the oracle's
own definition (see rope3d's docstring).
"""
from . import attention, int8_codec, ring_cache, rope3d, sparse

__all__ = ["attention", "int8_codec", "ring_cache", "rope3d", "sparse"]
