"""GB300-native SnapStream fixed-size KV cache (see include/snap.h for the C ABI)."""
