"""GB300-native routed MoE expert layer (binding placeholder)."""
