"""Groupwise int4/int5 weight-only dequant-GEMM for GB300 (sm_103a)."""
