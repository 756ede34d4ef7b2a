"""GB300-native (sm_103a) int8 quantized linear layer for LLM.int8-style
8-bit training: the memory-efficient ``Linear8bitLt`` of bitsandbytes PR #33
"Memory efficient backward".

    from int8_quantized_linear_i8lt_gb300 import Linear8bitLt
    layer = Linear8bitLt.from_float(weight, bias, threshold=6.0)
    y = layer(x)            # int8 forward with the fp16 outlier decomposition
    y.sum().backward()      # grad to x and to the bias; the weight is frozen

``LinearNF4`` / ``LinearFP4`` are the frozen 4-bit (NormalFloat / E2M1) layers
of QLoRA fine-tuning (bf16 or fp16 compute, the weight decoded inside the
tensor-core matmuls).

The arithmetic runs in libi8lt.so (hand-written CUDA for sm_103a, C ABI in
include/i8lt.h); build it with ``python -m int8_quantized_linear_i8lt_gb300.build``.
"""
from .functional import (I8LTError, Int8LinearFunction, Int8LinearTrainableFunction, Int8MLPFunction,
                         Linear4bitFunction, NF4LinearFunction, SiLUFunction, backward_input, backward_input_4bit,
                         default_max_outliers, dequantize_4bit, dequantize_absmax, device_status,
                         double_quantize_absmax, forward, forward_4bit,
                         fp4_backward_input, fp4_dequantize, fp4_forward, fp4_levels, fp4_quantize, grad_weight,
                         levels_4bit, nf4_backward_input, nf4_dequantize, nf4_forward, nf4_levels, nf4_quantize,
                         quantize_4bit, quantize_weight, silu, silu_backward, weight_ld)
from .module import Int8MLP, Linear4bit, Linear8bitLt, Linear8bitLtTrainable, LinearFP4, LinearNF4

__all__ = ["Linear8bitLt", "Linear8bitLtTrainable", "Int8MLP", "I8LTError", "Int8LinearFunction",
           "Int8LinearTrainableFunction", "Int8MLPFunction", "SiLUFunction", "forward", "backward_input",
           "grad_weight", "quantize_weight", "silu", "silu_backward", "device_status", "default_max_outliers",
           "weight_ld", "Linear4bit", "LinearNF4", "LinearFP4", "Linear4bitFunction", "NF4LinearFunction",
           "levels_4bit", "quantize_4bit", "dequantize_4bit", "forward_4bit", "backward_input_4bit",
           "nf4_levels", "nf4_quantize", "nf4_dequantize", "nf4_forward", "nf4_backward_input",
           "fp4_levels", "fp4_quantize", "fp4_dequantize", "fp4_forward", "fp4_backward_input",
           "double_quantize_absmax", "dequantize_absmax"]
