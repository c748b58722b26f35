"""GB300 (sm_103a) MoE expert layer: FP8 activations x FP4 weights with
counting-sort permute, tcgen05 block-scaled grouped GEMMs and a fused
SwiGLU (.) top-k-weight FP8 epilogue, behind a C ABI (include/moe_mxq.h);
and its block-FP8 variant (E4M3 weights with 128 x 128 float32 block
scales, include/moe_bfp8.h).

``binding`` holds the thin ctypes layer (same names as the C entry points);
``layer.MoELayer`` / ``layer.MoELayerBfp8`` own quantised weights and a
workspace for the fused ``moe_forward`` / ``moe_forward_bfp8`` calls.
"""
from . import binding  # noqa: F401  (raises ImportError if the library is not built)
from .binding import (MoeError, moe_combine, moe_expert_forward, moe_expert_workspace_size, moe_forward,  # noqa: F401
                      moe_get_device_status, moe_permute, moe_permute_workspace_size, moe_route_topk,
                      moe_status_string, moe_version, moe_workspace_size, mxq_quantize_act, mxq_quantize_weight,
                      bfp8_quantize_act, bfp8_quantize_weight, moe_bfp8_workspace_size, moe_forward_bfp8)
from .layer import Bfp8Experts, MoELayer, MoELayerBfp8, QuantizedExperts  # noqa: F401
