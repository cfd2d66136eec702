"""CPU oracle for the MoE expert FFN forward -- test infrastructure only.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may
import this package.  It shares no code with the CUDA library and never
imports it.  See ``oracle.moe_oracle`` for the definitions and their sources.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (bf16_round, e4m3_round, e4m3_decode, quantize_rows_e4m3, silu,  # noqa: F401
                         rms_norm, router_logits, softmax, topk_renorm, permute, silu_and_mul,
                         grouped_fc1, grouped_fc2, combine, moe_ffn_forward, ffn_token_outputs,
                         route, E4M3_MAX, BF16_MAX)
