"""float64 CPU oracle for speculative-decoding verification (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The CUDA path never does.
"""
from .spec_oracle import *  # noqa: F401,F403
from .spec_oracle import (SEQ_OK, SEQ_BAD_LENGTH, SEQ_BAD_TOKEN, SEQ_BAD_UNIFORM,  # noqa: F401
                          SEQ_NONFINITE, SEQ_EMPTY_SUPPORT, SEQ_ERROR_MASK,
                          SEQ_FLAG_ZERO_Q, SEQ_FLAG_Z_ZERO)
