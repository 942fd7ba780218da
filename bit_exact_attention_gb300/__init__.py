"""GB300-native SageAttention2 quantized attention forward (placeholder; binding added below)."""
