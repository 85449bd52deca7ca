"""GB300-native Llama-layout pre-norm decoder block (prefill and decode)."""
