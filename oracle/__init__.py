"""Float64 CPU oracle for the packed linear-attention pass and the packed
softmax-attention layer.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  It shares
no code with the CUDA library and never imports it.
"""
from .oracle import (  # noqa: F401
    build_oracle,
    oracle_pass,
    oracle_branches_from_state,
    oracle_max_threads,
    segment_quadratic,
    segment_chunked,
)
from .softmax_oracle import (  # noqa: F401
    oracle_softmax_pass,
    oracle_softmax_rows,
)
