"""GB300-native (sm_103a) MoE layer step of Kimi K3.

Router (sigmoid scores, correction-bias top-k), routed expert FFN read straight from
packed MXFP4, router-order combine and the shared expert -- in the direct layer and in
the pages' LatentMoE (latent projections, aggregate RMSNorm) -- as hand-written CUDA behind a
C ABI (``include/k3moe.h``, built into ``_build/libk3moe.so``); :mod:`.k3moe` is the
ctypes binding.  Importing the package does not load the library; the first call does,
and raises if it cannot.
"""
from .k3moe import (  # noqa: F401
    LayerDims, K3MoeError, k3moe_route, k3moe_expert_ffn_mxfp4, k3moe_layer,
    k3moe_layer_static_scratch, STATIC_SCRATCH_BYTES, k3moe_decode_stack,
    k3moe_rmsnorm_bf16, k3moe_dequant_mxfp4, k3moe_test_expire_wait, k3moe_trace_enable, k3moe_trace_read,
    record_layout, workspace_size, new_workspace, new_status, status_str, lib, EXPORTS,
    LatentDims, k3moe_latent_layer, latent_workspace_size, new_latent_workspace,
    ExpertCache, k3moe_layer_streamed, streamed_workspace_size, new_streamed_workspace,
)
