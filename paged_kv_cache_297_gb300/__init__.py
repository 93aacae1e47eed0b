"""GB300-native paged KV-cache attention (placeholder, binding added next)."""
