"""Exact attention forward pass for GB300 (sm_103a) behind a C-ABI library."""
