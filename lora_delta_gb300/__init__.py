"""GB300-native routed multi-tenant LoRA delta (placeholder during bring-up)."""
