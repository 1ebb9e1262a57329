"""GB300-native exact multi-head scaled dot-product attention (placeholder during bring-up)."""
