"""CPU oracle for the attention library -- TEST INFRASTRUCTURE ONLY.

``attention``: the FP64 definition (forward, backward, stabilised shift rule,
FP32 decidability bound).  ``emulation``: the FP32/BF16 (or FP8 P~) blocked
online-softmax forward.  ``fp8``: E4M3 encoding, per-tensor dynamic scaling and
the FP8 forward.  None of them shares code with the CUDA library; only the tests, the smoke
check and the benchmark's CPU-baseline leg may import this package.
"""
from . import attention, emulation, fp8  # noqa: F401
