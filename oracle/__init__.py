"""CPU oracle of the sparse MoE layer forward (test infrastructure only; see moe_oracle)."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import (e4m3_round, e4m3_value, quantize_fp8_rows, dequantize_fp8_rows, layer_forward_fp8, backward_dw_entries, backward_dx_tokens, Dispatch, ExpertChoice, Grads, Params, forward_fixed_routing, layer_backward, params64, LayerResult, expert_choice, expert_choice_forward, expert_choice_select, LoadStats, capacity, combine, dense_mask_forward, dispatch,  # noqa: F401
                         bias_update, expert_ffn, gate_weights, layer_forward, load_stats, router_logits, router_z_loss,
                         router_probabilities, selection_scores, sequence_balance_loss, sigmoid_affinity, silu, topk, widen)
