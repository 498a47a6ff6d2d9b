"""ORACLE — test infrastructure only.

A plain single-threaded C++ restatement of the ZeRO-1/2/3 step over a flat,
padded FlatParameter (``zero_oracle.cpp``), with a numpy-facing ctypes
wrapper.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The CUDA library never calls it
and shares no code with it.

Every function here is pinned by a ``-m "not gpu"`` test against what the
pages fix (printed values, closed forms, invariants, brute force); see the
header of ``zero_oracle.cpp`` for the passages followed and the readings
taken where the pages are silent.
"""

from .oracle import (  # noqa: F401
    Hyper,
    OracleLayout,
    accumulate,
    bf16_round,
    bf16_widen,
    build,
    clip_coef,
    dp_step,
    export_state,
    gather_unit,
    grad_norm,
    import_state,
    layout,
    library_path,
    make_master,
    nonfinite_count,
    reduce_element,
    state_bytes,
    step_scalars,
    step_window,
    zero3_backward_peak,
    zero_step,
)
