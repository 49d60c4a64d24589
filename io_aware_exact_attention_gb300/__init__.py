"""Exact tiled attention with online softmax for one GB300 (sm_103a)."""
