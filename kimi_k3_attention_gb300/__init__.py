"""GB300-native fused AttnRes + add2 + RMSNorm decode epilogue."""
