"""GB300-native (sm_103a) int8 quantized linear layer for LLM.int8-style
8-bit training: the memory-efficient ``Linear8bitLt`` of bitsandbytes PR #33
"Memory efficient backward".

    from int8_quantized_linear_i8lt_gb300 import Linear8bitLt
    layer = Linear8bitLt.from_float(weight, bias, threshold=6.0)
    y = layer(x)            # int8 forward with the fp16 outlier decomposition
    y.sum().backward()      # grad to x and to the bias; the weight is frozen

``LinearNF4`` is the frozen 4-bit NormalFloat layer of QLoRA fine-tuning
(bf16 or fp16 compute, the weight decoded inside the tensor-core matmuls).

The arithmetic runs in libi8lt.so (hand-written CUDA for sm_103a, C ABI in
include/i8lt.h); build it with ``python -m int8_quantized_linear_i8lt_gb300.build``.
"""
from .functional import (I8LTError, Int8LinearFunction, Int8LinearTrainableFunction, Int8MLPFunction,
                         NF4LinearFunction, SiLUFunction, backward_input, default_max_outliers, device_status, forward,
                         grad_weight, nf4_backward_input, nf4_dequantize, nf4_forward, nf4_levels, nf4_quantize,
                         quantize_weight, silu, silu_backward, weight_ld)
from .module import Int8MLP, Linear8bitLt, Linear8bitLtTrainable, LinearNF4

__all__ = ["Linear8bitLt", "Linear8bitLtTrainable", "Int8MLP", "I8LTError", "Int8LinearFunction",
           "Int8LinearTrainableFunction", "Int8MLPFunction", "SiLUFunction", "forward", "backward_input",
           "grad_weight", "quantize_weight", "silu", "silu_backward", "device_status", "default_max_outliers",
           "weight_ld", "LinearNF4", "NF4LinearFunction", "nf4_levels", "nf4_quantize", "nf4_dequantize",
           "nf4_forward", "nf4_backward_input"]
