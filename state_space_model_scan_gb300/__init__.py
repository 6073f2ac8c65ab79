"""GB300 (sm_103a) Mamba-2 SSD chunked scan.

The compute lives in libssd.so (C ABI, include/ssd.h); this package holds its
thin ctypes binding (``_lib``), convenience wrappers that allocate outputs and
workspace with torch (``api``), the seeded input generator (``inputs``) and the
build script (``build``).  Importing the package does not load the library; the
first call does, and raises if it has not been built.
"""
from .api import ssd_forward, ssd_backward, Workspace  # noqa: F401
