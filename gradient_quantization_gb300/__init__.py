"""AGoQ element-wise quantization path for GB300 (sm_103a): a C-ABI library
(libagoq.so, include/agoq.h) and its thin Python binding.

    from gradient_quantization_gb300 import agoq
    codes, scales = agoq.agoq_quant_act(x_bf16, bits=4)
"""
__version__ = "0.1.0"
