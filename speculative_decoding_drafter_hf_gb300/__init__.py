"""HyFlash drafter-layer hot path for GB300 (sm_103a).

The compute lives in libhyflash.so (C ABI in include/hyflash.h); this package
only marshals arguments to it. Build the library with
``python -m speculative_decoding_drafter_hf_gb300.build``. The binding names
below load on first use, so the build module stays importable before the
library exists; using any of them without the library raises ImportError.
"""
_BINDING_NAMES = ("EXPORTED", "Drafter", "Family", "HfBlockWeights", "HfConfig", "HfLayerWeights", "HyflashError",
                  "LIB_PATH", "Status", "Tensor", "make_config")

__all__ = list(_BINDING_NAMES)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError(name)
