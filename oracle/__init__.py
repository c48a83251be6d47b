"""CPU oracle for the attention library -- TEST INFRASTRUCTURE ONLY.

``attention``: the FP64 definition (forward, backward, stabilised shift rule,
FP32 decidability bound).  ``emulation``: the FP32/BF16 blocked online-softmax
forward.  Neither shares code with the CUDA library; only the tests, the smoke
check and the benchmark's CPU-baseline leg may import this package.
"""
from . import attention, emulation  # noqa: F401
