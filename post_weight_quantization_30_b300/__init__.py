"""GPTQ layer quantization (+ EoRA compensation, GPTQ-intrinsic LoRA) native to NVIDIA B300 (sm_103a).

The compute path is libgq.so (CUDA kernels behind a C ABI, include/gq.h); this
package is its thin Python binding.  Importing it loads the library and fails
if the library has not been built.
"""
from ._lib import (  # noqa: F401
    GQError,
    LIB_PATH,
    SIGNATURES,
    eora_compensate,
    gptq_bidup,
    gptq_code_decisions,
    gptq_factor,
    gptq_hessian_accumulate,
    gptq_intrinsic_lora,
    gptq_lora_basis,
    gptq_packed_linear,
    gptq_pack,
    gptq_quantize_layer,
    gptq_quantize_layer_noalloc,
    gptq_quantize_rtn,
    gptq_sweep,
    gptq_unpack,
    gptq_weight_error,
    gq_check_device,
    kernel_timing,
    lib,
)
