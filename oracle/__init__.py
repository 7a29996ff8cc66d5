"""CPU oracle for the paged KV cache hot path (TEST INFRASTRUCTURE ONLY).

Two independent restatements of the same definitions, both in fp64:

* ``oracle.np_oracle`` -- numpy, one gather + softmax per sequence and KV head;
* ``oracle.c_oracle``  -- plain C loops (``pagedkv_oracle.c``), loaded with
  ctypes, optionally threaded over sequences; also the timed CPU baseline.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  It imports nothing from the CUDA
library's package, and the CUDA library imports nothing from here.
"""

from . import np_oracle  # noqa: F401
