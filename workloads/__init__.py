"""Seeded synthetic workloads for the token-sparse MLA forward.

This package only draws random inputs (queries, a paged latent KV cache, block
tables, per-token top-k slot lists, the parts of split lists, value up-projection weights,
position lists and per-head q/K/V of the masked dense route) and packs them into the layouts the
kernel and the oracle read.  It contains none of the attention arithmetic, so
both sides of every parity check can take their inputs from here.
"""

from .configs import CONFIGS, WorkloadConfig, config_by_name
from .generators import (
    Workload,
    causal_position_lists,
    gathered_bytes,
    make_masked_dense_inputs,
    make_merge_parts,
    make_v_up_weights,
    make_workload,
    pad_heads,
    quantize_fp8_rows,
    split_lists,
)

__all__ = [
    "CONFIGS",
    "WorkloadConfig",
    "config_by_name",
    "Workload",
    "causal_position_lists",
    "gathered_bytes",
    "make_masked_dense_inputs",
    "make_merge_parts",
    "make_v_up_weights",
    "make_workload",
    "pad_heads",
    "quantize_fp8_rows",
    "split_lists",
]
