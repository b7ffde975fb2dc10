"""CPU oracle of the PowerSGD compression step -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does.
"""
from .powersgd import (  # noqa: F401
    Compressed, OracleState, StepOut, compress, data_sent_per_step, gram_schmidt,
    q_init, splitmix64_mix, splitmix64_stream, uniform_open0,
)
