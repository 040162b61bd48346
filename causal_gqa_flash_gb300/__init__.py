"""Causal grouped-query flash attention (forward and backward) for GB300 / sm_103a."""
