"""Packed speculative-verification attention and margin/accept for GB300 (sm_103a)."""
