"""CPU oracle of the MoE-layer forward pass (test infrastructure only).

Imported by the tests, the package smoke check and the benchmark's CPU
baseline; never by the product path.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import OracleResult, moe_forward  # noqa: F401
