"""CPU oracle of grouped MoE prefill (test infrastructure; see moe_oracle)."""

from . import moe_oracle

__all__ = ["moe_oracle"]
