"""Float64 CPU oracle for the sparse-MoE layer (test infrastructure only).

Importable from the test suite, the smoke check and the benchmark's CPU
baseline leg; never from the CUDA library path.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (f64, router_logits, topk_indices, topk_mask, softmax, gating, silu,
                         expert, moe_layer, moe_layer_dense, moe_layer_tokens, permutation,
                         rmsnorm, moe_block, logit_gaps, Gating, LayerResult, Permutation,
                         RMS_EPS, LayerGrads, dsilu, moe_layer_backward)
from . import fp8_oracle  # noqa: F401
from .fp8_oracle import (e4m3_decode, e4m3_encode, quantize_weight_columns, dequantize_weight_columns,  # noqa: F401
                         quantize_rows, dequantize_rows, moe_layer_fp8, E4M3_MAX)
