"""GB300-native Kimi Delta Attention (KDA) forward."""
