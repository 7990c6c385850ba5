"""DynaSpec draft head + speculative-sampling verification for GB300 (sm_103a).

The compute lives in ``libdynaspec.so`` (hand-written CUDA behind the C ABI declared in
``include/dynaspec.h``).  ``api`` marshals torch tensors into those calls; ``pipeline``
strings them into one chain or tree speculation step with the router on a side stream.
"""
from . import _lib
from ._lib import DynaSpecError

__all__ = ["api", "pipeline", "DynaSpecError", "load_library"]


def load_library():
    """Load the CUDA library; raises ImportError if it has not been built."""
    return _lib.load()


from . import api        # noqa: E402
from . import pipeline   # noqa: E402
