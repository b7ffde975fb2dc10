"""GB300-native PowerSGD compression step.

The compute lives in ``libpsgd.so`` (hand-written CUDA for sm_103a, C ABI in
``include/psgd.h``); this package only builds it and binds it with ctypes.
"""
from .binding import (  # noqa: F401
    EXPORTS, LIB_PATH, PHASES, PSGD_ERR_CUDA, PSGD_ERR_INVALID, PSGD_ERR_OOM, PSGD_ERR_STATE, PSGD_ERR_TIMEOUT,
    PSGD_OK, PSGD_POWERSGD, PSGD_RTOPK,
    PowerSGD, PsgdError, lib, psgd_count_sent, psgd_plan_layout, psgd_plan_one_pass, psgd_plan_queue, step_noalloc,
)
from .build import build  # noqa: F401
