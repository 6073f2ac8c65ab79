"""Float64 CPU oracle for the Mamba-2 SSD scan -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product (``state_space_model_scan_gb300``) never
imports it, and it imports nothing from the product.

Contents
--------
``sequential``  ctypes front-end of ``ssd_oracle.c``: the literal O(T) loop over
                time and its exact adjoint (float64).
``quadratic``   the materialised semiseparable (closed) form, NumPy float64.
``chunked64``   the chunkwise decomposition (intra-chunk segment sums + carried
                chunk states), NumPy float64.

Parity status of each function is recorded in its module docstring.
"""
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssd_oracle.so")
SRC_PATH = os.path.join(_HERE, "ssd_oracle.c")


def build(force: bool = False) -> str:
    """Compile ``ssd_oracle.c`` into ``libssd_oracle.so`` (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC_PATH):
        return LIB_PATH
    tmp = LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", SRC_PATH, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH
