"""GPTQ per-layer quantization solver for NVIDIA B300 (sm_103a)."""
