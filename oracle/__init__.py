"""CPU oracle of grouped MoE prefill (test infrastructure): C++ in moe_oracle.cpp, marshalled by moe_oracle."""

from . import moe_oracle

__all__ = ["moe_oracle"]
