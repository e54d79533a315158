"""Packed linear-attention pass for GB300 (sm_103a)."""
