"""GB300-native W2A8 ternary matmul (BitNet b1.58 i2_s layout).

The CUDA library is loaded on first use by ``ternary_weight_gb300.binding``.
"""
