"""Seeded synthetic inputs for the MoE layer (shared by tests, smoke and bench).

This package draws the random tensors and turns the drawn fp32 expert weights
into the 4-bit formats the layer consumes. It holds none of the layer's own
arithmetic (routing, alignment, dequantisation, GEMMs, activation, reduce):
quantising the drawn weights is how the synthetic inputs are made (each
workload is "drawn fp32 N(0, 0.02), then quantised"), and both the CUDA path
and the CPU oracle read the same quantised bytes.
"""
from .configs import CONFIGS, get_config  # noqa: F401
from .gen import make_layer, to_numpy  # noqa: F401
