"""GB300-native Gated DeltaNet layer hot path (placeholder; binding added with the library)."""
