"""GB300 (sm_103a) latent-MoE layer forward: CUDA kernels behind a C ABI.

The Python names mirror the C entry points of include/lmoe.h; they only
marshal torch tensors (device memory, streams) into the library.
"""
from ._binding import (  # noqa: F401
    ABI_FUNCTIONS, LIB_PATH, LmoeDebug, LmoeDims, LmoeError, LmoeWeights, latent_moe_forward, latent_moe_forward_noalloc,
    latent_moe_forward_routed,
    latent_moe_launch_count, latent_moe_workspace_offsets, NUM_STAGES, STAGE_NAMES, WS_NAMES,
    latent_moe_workspace_bytes, lmoe_abi_version, lmoe_linear, lmoe_device_error, load_library, make_dims,
    make_weights, masked_situ_and_mul, moe_route, situ_and_mul, status_string, gemm_unit_walk,
    lmoe_router_logits, lmoe_router_logits_workspace_bytes, latent_moe_forward_router,
    latent_moe_launch_count_router, LmoeMxfp4Experts, lmoe_dequant_mxfp4, make_mxfp4_experts,
    latent_moe_workspace_bytes_mxfp4, latent_moe_forward_mxfp4, latent_moe_launch_count_mxfp4,
)
