"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or calls it, and this package imports
nothing from the product.  The arithmetic lives in ``oracle.c``; this module only
builds that file with gcc and marshals numpy arrays into it.
"""
from .oracle import (  # noqa: F401
    build,
    default_threads,
    fwd,
    fwd_blockwise,
    fwd_rows,
    bwd,
    bwd_rows,
    online_row,
    BF16,
    F64,
)
