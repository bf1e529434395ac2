"""Oracle package: plain fp64 CPU definitions of the vocabulary-sharded
embedding and the globally normalised cross-entropy.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers. The CUDA path never imports
this package and this package never imports the CUDA path.
"""
from . import vce_oracle  # noqa: F401
