"""Deterministic, batch-invariant linear-layer GEMM for GB300 (sm_103a)."""
