"""GB300-native split-KV decode attention with an intra-GPU log-sum-exp tree combine."""
