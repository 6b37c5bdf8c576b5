"""GB300-native dequantize-fused quantized matmul (GPTQ 4-bit and EXL2).

The compute path is the C-ABI library ``libexq.so`` (CUDA kernels for
sm_103a plus C++ host packers); ``exq`` is its ctypes binding. Build it with
``python quantized_weight_exq_gb300/build.py`` or ``__graft_entry__.build()``.
"""
from .exq import *  # noqa: F401,F403
from .exq import Weight, exl2_weight, gptq_weight, library_path  # noqa: F401
