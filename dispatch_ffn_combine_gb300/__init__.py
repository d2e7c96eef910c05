"""GB300-native fused MoE layer: route -> dispatch -> grouped SwiGLU FFN -> combine."""
