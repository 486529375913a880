"""Offline code generator for the per-class ERI kernels (see eri_gen.py)."""
