"""XAttention block-sparse chunked prefill for GB300 (sm_103a)."""
