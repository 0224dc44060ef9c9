"""CPU oracle for the quantized linear layer Y = X·Wᵀ.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the GPU path computes.  It exists to check the CUDA
library, never to stand in for it: only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference leg may import it.  The product
path (``quantized_linear_layer_gb300``) never imports it and shares no code,
table or constant with it.

Sources (the five web pages the method is taken from):

* "Chapter 9 - Quantization kernels: INT8 / FP8 / INT4" (a CUDA engineering
  book, yangyitao.com) - sections 9.2 (affine quantization), 9.6 (INT4 unpack).
* "LLM and AIGC quantization: from number formats to W4A4" (valdrada.cn) -
  sections on integers, floating point, block-scaled formats, linear
  quantization, symmetric/asymmetric, granularity, W8A8 integer GEMM, W4A16,
  and the AWQ offline flow (``pseudo_quant``).
* "vLLM W8A8 quantized GEMM: CUTLASS epilogue design" (blog.gitcode.com) -
  sections 2 (linear algebra), 2.1-2.4 (the four epilogues), 3 (evaluation
  order), 5 (azp_adj precompute).
* "NVFP4 quantization and ARCQuant" (lpnh.cn) - sections 2.1 (residual channel
  augmentation), 2.2 (augmented GEMM).

Arithmetic conventions: every quantizer works in float32 with IEEE
round-to-nearest operations exactly as written (numpy performs each float32
operation separately; nothing is fused), rounds to integers with
round-half-to-even (``np.rint``), and divides rather than multiplying by a
reciprocal.  GEMM results are formed in float64 from exactly dequantized
operands; integer GEMMs are exact.

Parity status per function is recorded in each module's header.
"""

from .formats import (  # noqa: F401
    E2M1_MAGNITUDES,
    e2m1_decode,
    e2m1_encode,
    e4m3_decode,
    e4m3_encode,
    e4m3_finite_magnitudes,
    int4_decode,
    pack_u4,
    unpack_u4,
)
from .quant import (  # noqa: F401
    quantize_affine,
    dequantize_affine,
    quant_sym_rows,
    quant_int8_sym,
    quant_int8_asym,
    quant_w4_g128,
    quant_fp8_rows,
    quant_fp8_tensor,
    sum_squares_f32,
    rmsnorm_rows,
    rmsnorm_quant_int8,
    rmsnorm_quant_fp8,
    rmsnorm_arc_quantize_activation,
    nvfp4_global_scale,
    nvfp4_quantize,
    nvfp4_dequantize,
    arc_perm,
    arc_quantize_activation,
    arc_quantize_weight,
)
from .mx import (  # noqa: F401
    MX_BLOCK,
    MX_EMAX,
    mx_block_exponent,
    mx_quantize,
    mx_dequantize,
    mx_gemm_reference,
    e8m0_decode,
)
from .hadamard import (  # noqa: F401
    hadamard_rotate,
    sylvester_matrix,
    regular_matrix,
)
from .gemm import (  # noqa: F401
    w4a16_reference,
    w4a16_reference_packed,
    w4a16_act_order_reference,
    act_order_perm,
    int8_gemm_exact,
    azp_adj_from_weight,
    w8a8_epilogue,
    nvfp4_gemm_reference,
    fp8_gemm_reference,
)
