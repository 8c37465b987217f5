"""CPU oracle for exact, IO-aware, tiled attention (FlashAttention).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
anything from this package.  The GPU path (``exact_io_aware_tiled_gb300``) never
imports it, and this package imports nothing from the GPU path.

Everything here is plain numpy in float64, written to be checked against the
pages by eye rather than to be fast:

* ``attention``   -- the definition: materialise S and P, mask, softmax, dropout,
                     O = P~ V, and the backward by the chain rule.
* ``tiled``       -- the three tiled online-softmax loop orders the pages print
                     (KV-outer normalised every step; Q-outer normalised every
                     step; Q-outer with deferred normalisation), simulated on CPU.
* ``philox``      -- Philox4xW-R (Salmon et al., SC'11), generic over word width,
                     and the dropout keep-mask mapping used by the method.
* ``traffic``     -- instrumented HBM element counts of the naive and tiled
                     algorithms, for the pages' byte-accounting worked numbers.
* ``masks``       -- the causal / sliding-window / key-padding / block-sparse
                     mask definitions.
* ``fp8``         -- the FP8 forward: E4M3 rounding, the random Hadamard
                     rotation, block (or per-tensor) quantisation and the
                     online-softmax forward on the quantised inputs.

Parity status of each function is stated in its own docstring ("pinned by ...").
"""
from . import philox, masks, attention, tiled, traffic, fp8  # noqa: F401
