"""DFlash 2 draft-selection + verify path on one GB300 (sm_103a).

The compute runs in ``libdflash2.so`` (hand-written CUDA behind the C ABI of
``include/dflash2.h``); ``dflash2`` below is a thin binding that only
marshals torch tensors into pointers.  Importing this package loads nothing;
the first call loads the library and raises if it is missing.
"""
from .binding import (  # noqa: F401
    DFlash2Error,
    Workspace,
    conv2tap,
    ctx_gate,
    device_error,
    dynconv2tap,
    lmhead_topk16,
    load_library,
    pair_score_walk,
    sampling_params,
    test_hold,
    topk16,
    topk16_merge,
    topk16_noalloc,
    topk16_shard,
    verify,
)
