"""CPU oracle for the RDKV hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the ``rdkv_*`` C-ABI library and its Python binding) never calls it, and it
shares no code, table or constant generator with the CUDA sources.

Parity status of each function is stated in ``rdkv_oracle``'s module header.
"""
from .rdkv_oracle import *  # noqa: F401,F403
