"""GB300-native RMSNorm forward/backward (plain and fused-add)."""
