"""libvocabce for GB300: vocabulary-sharded embedding lookup and globally
normalised cross-entropy over a padded vocabulary, as hand-written sm_103a
CUDA behind a C ABI (include/vce.h).

``vocab_embedding_cross_gb300.vce`` is the ctypes binding (same names as the C
entry points); it is loaded on first use and raises if the library has not
been built. ``inputs`` draws the seeded synthetic workloads.
"""
from . import inputs  # noqa: F401


def __getattr__(name):
    if name == "vce":
        from . import _lib
        return _lib
    raise AttributeError(name)
