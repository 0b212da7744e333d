"""CPU oracle (float64 NumPy) for QK-RMSNorm joint attention — test infrastructure only."""
from .jattn_oracle import (EPS, attention_bwd_head, attention_fwd_head, attention_one_row, joint_attention_bwd,
                           joint_attention_fwd, joint_attention_streams, joint_attention_varlen_bwd, qkv_norm_streams,
                           qkv_projection, rmsnorm_bwd, rmsnorm_fwd, round_to_bf16)
