"""GB300-native GPTQ per-layer quantization: a C-ABI CUDA library plus a thin binding."""
