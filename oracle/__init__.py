"""CPU oracle for the HyFlash drafter layer -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct NumPy float64 code that states what one drafter
layer computes. Only the tests, the smoke check and the benchmark's CPU
baseline / reference arm may import it; the product path never does. It
shares no code with the CUDA library and imports nothing from it.

Parity status per function is listed in ``oracle.hyflash_oracle.__doc__``.
"""
from .hyflash_oracle import *  # noqa: F401,F403
