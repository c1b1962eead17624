"""Barrier-free small-message AllReduce over N virtual ranks on one GB300.

Importing the package does not load the CUDA library; ``rra`` loads it on
first use and raises if it is missing (there is no CPU fallback).
"""
__all__ = ["rra", "inputs"]
