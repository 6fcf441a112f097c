"""Fused linear cross-entropy for GB300 (sm_103a): a thin binding over ``libflce.so``."""
