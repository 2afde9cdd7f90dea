"""GB300-native MoE expert-parallel dispatch / combine (placeholder, filled below)."""
