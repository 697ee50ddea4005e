"""GB300-native LM-head contraction fused with the consumer-surface projection."""
