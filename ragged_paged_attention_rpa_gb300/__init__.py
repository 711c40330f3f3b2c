"""Ragged paged attention for one GB300 (sm_103a)."""
