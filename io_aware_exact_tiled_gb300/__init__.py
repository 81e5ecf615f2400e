"""Fused, tiled, exact softmax attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libfa.so`` built from ``csrc/``; the
Python layer only marshals arguments (see ``binding``).
"""
