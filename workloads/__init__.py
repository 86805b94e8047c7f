"""Seeded synthetic inputs for grouped MoE prefill.

This package only draws random inputs (router logits, token rows, expert
weights, the owner mask).  It computes nothing that the MoE path computes, so
both the CPU oracle and the CUDA path can consume its output without sharing
any of the method's arithmetic.
"""

from .synthetic import CONFIGS, MoEConfig, make_inputs, make_logits, make_mask, make_tokens, make_weights

__all__ = ["CONFIGS", "MoEConfig", "make_inputs", "make_logits", "make_mask", "make_tokens", "make_weights"]
