"""The oracle: a plain, slow CPU reference of the conv + BN + activation backward.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  The product path (the
CUDA library and its binding) never imports it.

Every value is computed in double precision by ``cba_ref.c``; ``ref.py`` holds
the ctypes wrappers that take numpy arrays.
"""
from .ref import *  # noqa: F401,F403
