"""OSCAR 2-bit KV-cache hot path for GB300 (sm_103a): package root."""
