"""Ragged paged attention for one GB300 (sm_103a).

The computation lives in ``librpa.so`` (C ABI declared in ``include/rpa.h``,
CUDA kernels under ``csrc/``).  This package holds its build step
(``build.py``), a thin ctypes binding with the same entry-point names
(``binding.py``) and the seeded synthetic workloads (``workloads.py``).
Importing the package loads nothing; the first library call loads librpa.so
and raises if it has not been built.
"""

from .binding import (  # noqa: F401
    RPA_DTYPE_BF16, RPA_DTYPE_F32, RPA_PATH_AUTO, RPA_PATH_SIMT, RPA_PATH_TC,
    RPA_DEVERR_NONE, RPA_DEVERR_PAGE_ID, RPA_DEVERR_LENGTHS, RPA_DEVERR_PLAN,
    RPA_DEVERR_TIMEOUT, Batch, ForwardCall, Plan, RpaError, alloc_workspace, rpa_clear_device_error,
    rpa_forward, rpa_get_device_error, rpa_plan, rpa_status_string, rpa_trace_begin,
    rpa_trace_end)
