"""Seeded synthetic workloads shared by the oracle tests, the GPU tests and the bench."""
from .gen import (CONFIGS, Config, HeadStream, LayerData, denoise_steps, layer_data, planes, prompt, round_bf16,
                  to_storage)

__all__ = ["CONFIGS", "Config", "HeadStream", "LayerData", "denoise_steps", "layer_data", "planes",
           "prompt", "round_bf16", "to_storage"]
