"""vocab_ce_gb300 -- Megatron-style 1D tensor-parallel MLP block and
vocabulary-parallel fused cross-entropy, all t shards on one GB300 (sm_103a).

The compute lives in the CUDA library ``lib/libtpce.so`` (C ABI in
``include/tpce.h``); this package only marshals torch tensors to it.
"""

from .api import (TpceError, attn_workspace_bytes, tp_attn_out_backward_sp, tp_attn_out_forward_sp,
                  tp_attn_qkv_backward_sp, tp_attn_qkv_forward_sp, tp_column_linear_backward_sp,
                  tp_column_linear_forward_sp, tp_row_linear_backward_sp, tp_row_linear_forward_sp, ce_workspace_bytes, device_status, device_status_detail,
                  linear_workspace_bytes, mlp_workspace_bytes, pad_vocab, profile_enable, profile_read,
                  swiglu_workspace_bytes, tail_workspace_bytes, tp_attn_out_backward, tp_attn_out_forward, tp_attn_qkv_backward,
                  tp_attn_qkv_forward, tp_linear_backward, tp_linear_forward, tp_mlp_backward, tp_mlp_backward_sp,
                  tp_mlp_forward, tp_mlp_forward_sp, tp_swiglu_backward, tp_swiglu_backward_sp, tp_swiglu_forward,
                  tp_swiglu_forward_sp, vocab_parallel_ce, vocab_parallel_ce_loss_static)

__all__ = ["TpceError", "attn_workspace_bytes", "tp_attn_out_backward_sp", "tp_attn_out_forward_sp",
           "tp_attn_qkv_backward_sp", "tp_attn_qkv_forward_sp", "tp_column_linear_backward_sp",
           "tp_column_linear_forward_sp", "tp_row_linear_backward_sp", "tp_row_linear_forward_sp", "ce_workspace_bytes", "device_status", "device_status_detail",
           "linear_workspace_bytes", "mlp_workspace_bytes", "pad_vocab", "profile_enable", "profile_read",
           "swiglu_workspace_bytes", "tail_workspace_bytes", "tp_attn_out_backward", "tp_attn_out_forward", "tp_attn_qkv_backward",
           "tp_attn_qkv_forward", "tp_linear_backward", "tp_linear_forward", "tp_mlp_backward", "tp_mlp_backward_sp",
           "tp_mlp_forward", "tp_mlp_forward_sp", "tp_swiglu_backward", "tp_swiglu_backward_sp", "tp_swiglu_forward",
           "tp_swiglu_forward_sp", "vocab_parallel_ce", "vocab_parallel_ce_loss_static"]
