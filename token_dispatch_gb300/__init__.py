"""GB300-native MoE / MoD layer hot path: a C-ABI CUDA library (libmoe) and a
thin Python binding over it."""
