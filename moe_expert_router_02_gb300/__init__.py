"""Fused MoE router for NVIDIA GB300 (sm_103a).

The compute path is the CUDA library ``libgbrouter.so`` (C ABI in
``include/gbrouter.h``); :mod:`.router` is its Python binding and
:mod:`.synth` builds seeded synthetic inputs.
"""
