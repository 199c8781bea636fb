"""GB300-native paged GQA attention (KV append, batched decode, chunked prefill)."""
