"""Tree-verify step for tree speculative decoding on GB300 (sm_103a)."""
