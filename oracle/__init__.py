"""CPU oracle for the MoE layer hot path (test infrastructure only; see moe_oracle)."""
from . import moe_oracle  # noqa: F401
