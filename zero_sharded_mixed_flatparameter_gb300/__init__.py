"""GB300 (sm_103a) ZeRO-1/2/3 optimizer step over a flattened, padded FlatParameter.

The compute path is the CUDA library ``libzero_flatstep.so`` behind the C ABI
of ``include/zero_flatstep.h``; :mod:`.binding` marshals its calls and
:mod:`.runner` allocates the caller's device buffers with torch.
"""

from . import binding  # noqa: F401
from .binding import ZeroError  # noqa: F401


def build(force: bool = False, verbose: bool = False) -> str:
    from .build_lib import build as _build
    return _build(force=force, verbose=verbose)
