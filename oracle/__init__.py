"""CPU oracle for absorbed-MLA decode — TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 restatement of what the pages define (naive expand-then-
attend and the absorbed form), plus the fp32 cache quantizers.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA library and the
product package never imports it.
"""

from .mla_oracle import *  # noqa: F401,F403
