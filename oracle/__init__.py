"""CPU oracle for the speculative-decoding verification step.

Test infrastructure only: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline legs of ``bench.py``; never by the library.
"""
from .oracle import *  # noqa: F401,F403
from .oracle import NEAR_TIE, verify_request, greedy_request, verify_batch, greedy_batch  # noqa: F401
