"""CPU oracle for the owner-side Muon update (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library itself never calls it and
shares no code with it.
"""
from .ns_oracle import (  # noqa: F401
    EPS, QUINTIC, CUBIC,
    momentum_update, orient, frob_normalize, ns_original, ns_gram,
    newton_schulz, muon_update, bf16_round, bucket_order,
)
from . import partition  # noqa: F401,E402
from . import adamw  # noqa: F401,E402
