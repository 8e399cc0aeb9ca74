"""Orca-style iteration-level scheduling with selective batching on one GB300.

The package has three layers:

* ``synth``   -- seeded synthetic inputs (model weights, request traces, cached
  K/V contents).  It holds none of the method's arithmetic and is the only
  module shared with the CPU oracle used by the tests.
* ``native``  -- the ctypes binding of ``liborca.so`` (the C ABI declared in
  ``include/orca.h``): engine, K/V reservation pool and iteration-level
  scheduler.  Argument marshalling only; every step of the hot path runs in the
  library's CUDA kernels.
* ``build``   -- compiles ``liborca.so`` for sm_103a with nvcc.

Importing the package does not load the CUDA library; ``native`` does, and it
raises if the library has not been built.
"""

__all__ = ["synth", "native", "build"]
