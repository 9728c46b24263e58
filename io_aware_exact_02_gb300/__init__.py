"""GB300-native exact, IO-aware fused attention.

The compute lives in the C-ABI library ``libfa.so`` (hand-written CUDA for
sm_103a); :mod:`io_aware_exact_02_gb300.fa` is its thin ctypes binding and
:mod:`io_aware_exact_02_gb300.synth` draws the seeded synthetic inputs.
Importing the package loads nothing; the library is loaded on first use and
a missing or unloadable library raises.
"""
