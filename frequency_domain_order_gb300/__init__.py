"""GB300-native frequency-domain overlap-save FIR filtering.

``fir_os`` is the Python binding of libfir_os.so (C ABI in include/fir_os.h); ``build``
compiles it in-tree for sm_103a.  Importing this package loads nothing; the library is loaded
on first use and its absence is an error, never a fallback.
"""
from . import fir_os  # noqa: F401
from .fir_os import Plan, FirOsError  # noqa: F401
