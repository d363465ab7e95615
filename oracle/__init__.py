"""Float64 CPU oracle for the sparse-MoE layer (test infrastructure only).

Importable from the test suite, the smoke check and the benchmark's CPU
baseline leg; never from the CUDA library path.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (f64, router_logits, topk_indices, topk_mask, softmax, gating, silu,
                         expert, moe_layer, moe_layer_dense, moe_layer_tokens, permutation,
                         rmsnorm, moe_block, logit_gaps, Gating, LayerResult, Permutation,
                         RMS_EPS)
