"""Seeded synthetic workloads for the MoE FFN forward pass (inputs only, no MoE arithmetic)."""
from .generator import (WORKLOADS, MoEShape, TENSOR_IDS, bf16_round, bf16_to_f32, to_f64,
                        gen_x, gen_router, gen_logit_bias, gen_sel_bias, gen_expert, gen_experts,
                        expert_dims, gen_matrix, standard_normal, workload_arrays)

__all__ = ["WORKLOADS", "MoEShape", "TENSOR_IDS", "bf16_round", "bf16_to_f32", "to_f64",
           "gen_x", "gen_router", "gen_logit_bias", "gen_sel_bias", "gen_expert", "gen_experts",
           "expert_dims", "gen_matrix", "standard_normal", "workload_arrays"]
