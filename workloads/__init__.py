"""Seeded synthetic workloads (sizes and input tensors) for the VeriCache round."""
from .configs import (Workload, DROP, QUANT, ALL, by_index, scaled, tiny, llama8b_drop,  # noqa: F401
                      qwen32b_quant2, llama70b_offload4, mixed_serving)
from . import gen  # noqa: F401
