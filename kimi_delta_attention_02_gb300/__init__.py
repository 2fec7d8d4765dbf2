"""Kimi Delta Attention (KDA) prefill and decode for NVIDIA GB300 (sm_103a).

The compute lives in ``libkda.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/kda.h``). This package only marshals arguments to it
(``kimi_delta_attention_02_gb300.binding``) and generates seeded synthetic
inputs (``kimi_delta_attention_02_gb300.workloads``). There is no CPU fallback:
the binding raises if the library is missing.
"""
