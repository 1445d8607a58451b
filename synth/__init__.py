"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle's callers.

This package holds no arithmetic of the method: it only draws normal numbers, stores them as bf16
and copies rows to plant ties. Both the CUDA path and the oracle are fed from it.
"""
