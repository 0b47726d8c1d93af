"""Float64 CPU oracle of the dropless MoE layer (test infrastructure only).

Only tests, the package smoke check and the bench's CPU-baseline leg use it;
the CUDA product path never imports it."""

from .moe_oracle import *  # noqa: F401,F403
