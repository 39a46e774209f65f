"""Workload sizes and seeded synthetic inputs shared by the oracle and the CUDA path."""
from . import configs, synth  # noqa: F401
