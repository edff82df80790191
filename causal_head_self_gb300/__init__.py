"""GB300-native scaled dot-product causal multi-head self-attention."""
