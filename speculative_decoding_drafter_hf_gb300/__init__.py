"""HyFlash drafter-layer hot path for GB300 (sm_103a).

The compute lives in libhyflash.so (C ABI in include/hyflash.h); this package
only marshals arguments to it. Build the library with
``python -m speculative_decoding_drafter_hf_gb300.build``.
"""
from ._binding import (  # noqa: F401
    EXPORTED,
    Drafter,
    Family,
    HfConfig,
    HfLayerWeights,
    HyflashError,
    LIB_PATH,
    Status,
    Tensor,
    make_config,
)
