"""OSCAR CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  It wraps ``oscar_oracle.cpp`` (plain fp64
C++, single-threaded) through ctypes; ``calibration.py`` holds the offline
calibration (covariance, spectral rotation, clipping thresholds) in fp64 numpy.
Neither shares anything with the CUDA library.
"""

from .oracle import *  # noqa: F401,F403
