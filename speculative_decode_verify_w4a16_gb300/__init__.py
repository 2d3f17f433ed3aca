"""GB300-native W4A16 speculative-verify hot path.

Exposes the C-ABI library libw4a16sv (CUDA kernels for sm_103a) through a thin
torch-tensor binding:
  quantize, prepack, PackedWeight, linear      -- the W4A16 verify linear
  linear_logits                                -- the lm_head with fused softmax statistics
  spec_accept, spec_accept_prestat,
  spec_accept_node                             -- the speculative accept step
  tree_attention, kv_compact                   -- tree-masked verify attention, accepted-path KV compaction
  check_device_status                          -- device error word
"""
from .api import (PackedWeight, accept_workspace_bytes, check_device_status, kv_compact, linear, linear_logits,
                  linear_logits_workspace_bytes, linear_noalloc, linear_workspace_bytes, packed_scale_bytes,
                  packed_weight_bytes, prepack, quantize, spec_accept, spec_accept_node, spec_accept_prestat,
                  tree_attention, tree_attention_workspace_bytes, workspace)
from ._lib import LIB_PATH, W4A16Error, lib, status_string

__all__ = [
    "PackedWeight", "accept_workspace_bytes", "check_device_status", "kv_compact", "linear", "linear_logits",
    "linear_logits_workspace_bytes", "linear_noalloc", "linear_workspace_bytes", "packed_scale_bytes",
    "packed_weight_bytes", "prepack", "quantize", "spec_accept", "spec_accept_node", "spec_accept_prestat",
    "tree_attention", "tree_attention_workspace_bytes", "workspace",
    "LIB_PATH", "W4A16Error", "lib", "status_string",
]
