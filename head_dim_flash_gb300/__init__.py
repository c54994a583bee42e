"""Exact softmax attention for large head dims (D = 320..1024) on GB300 (sm_103a)."""
