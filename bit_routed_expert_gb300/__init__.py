"""GB300-native routed-expert MoE layer and Engram gather-decode (libbre, sm_103a).

The compute path is the C-ABI library built from ``csrc/`` (see ``include/bre.h``);
this package holds its Python binding (``api``), the build step (``build``) and the
seeded synthetic-input generator (``synth``).
"""
from .api import (FfnWeights, MoeLayer, MoeStack, StepGraph, bre_dequant, engram_gather_decode, engram_inject, engram_inject_workspace, moe_combine, moe_expert_ffn,
                  moe_expert_ffn_workspace, moe_permute, moe_residual_norm, moe_route, moe_route_ex, moe_route_permute,
                  moe_route_workspace)
from ._lib import BRE_FMT_Q2_K, BRE_FMT_Q8_0, BreError, load

__all__ = ["FfnWeights", "MoeLayer", "MoeStack", "StepGraph", "bre_dequant", "engram_gather_decode", "engram_inject", "engram_inject_workspace", "moe_combine", "moe_expert_ffn",
           "moe_expert_ffn_workspace", "moe_permute", "moe_residual_norm", "moe_route", "moe_route_ex", "moe_route_permute",
           "moe_route_workspace",
           "BRE_FMT_Q2_K", "BRE_FMT_Q8_0", "BreError", "load"]
